// Register-only throughput of the DP relaxation's arithmetic: the denominator of
// the sweep's roofline.  The min-max recurrence of Nest (Network- and Memory-Aware
// Device Placement) §4 Eq. 3 tries every candidate (j, m, c') against every cell.
// On plain words one such relaxation is one max (the stage load against the
// remaining pipeline), one compare against the cell's running best and two selects
// (value and argument); on tagged 32-bit words (the width index in the low bits, so
// no argument travels with the value) it is one max and one min.  This kernel
// issues one of those mixes on values held in registers, with four independent
// running bests per thread and full occupancy.  Every (candidate, running best) pair
// has its own max operands and the candidates' values move by one add per iteration,
// so no max is loop-invariant or shared (the assembler would hoist or merge those);
// the adds cost 1/4 of an operation per relaxation, so the figure is slightly below
// the mix's own peak.  It is measurement infrastructure, loaded only by bench.py.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kThreads = 512;
constexpr int kCand = 8;   // candidates kept in registers
constexpr int kAcc = 4;    // independent running bests per thread

__device__ __forceinline__ uint32_t vmax(uint32_t a, uint32_t b) {
    uint32_t r;
    asm volatile("max.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint64_t vmax(uint64_t a, uint64_t b) {
    uint64_t r;
    asm volatile("max.s64 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ void keep_min(uint32_t v, uint32_t idx, uint32_t &bv, uint32_t &bi) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.u32 p, %2, %0;\n\tselp.b32 %0, %2, %0, p;\n\tselp.b32 %1, %3, %1, p;\n\t}"
                 : "+r"(bv), "+r"(bi)
                 : "r"(v), "r"(idx));
}
__device__ __forceinline__ void keep_min(uint64_t v, uint32_t idx, uint64_t &bv, uint32_t &bi) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.s64 p, %2, %0;\n\tselp.b64 %0, %2, %0, p;\n\tselp.b32 %1, %3, %1, p;\n\t}"
                 : "+l"(bv), "+r"(bi)
                 : "l"(v), "r"(idx));
}

__device__ __forceinline__ void keep_min_tagged(uint32_t v, uint32_t &bv) {
    asm volatile("min.u32 %0, %0, %1;" : "+r"(bv) : "r"(v));
}

template <typename V, bool kTagged>
__global__ void __launch_bounds__(kThreads) peak_kernel(int iters, uint32_t seed, unsigned long long *sink) {
    V a[kCand], n[kAcc];
    uint32_t x = seed ^ (blockIdx.x * kThreads + threadIdx.x) * 2654435761u;
#pragma unroll
    for (int m = 0; m < kCand; m++) {
        x = x * 1664525u + 1013904223u;
        a[m] = V(x >> 8);
    }
#pragma unroll
    for (int q = 0; q < kAcc; q++) {
        x = x * 1664525u + 1013904223u;
        n[q] = V(x >> 8);
    }
    V bv[kAcc];
    uint32_t bi[kAcc];
#pragma unroll
    for (int q = 0; q < kAcc; q++) {
        bv[q] = V(0x7FFFFFFFu);
        bi[q] = 0xFFFFFFu;
    }
    for (int it = 0; it < iters; it++) {
#pragma unroll
        for (int m = 0; m < kCand; m++) {
#pragma unroll
            for (int q = 0; q < kAcc; q++) {
                if constexpr (kTagged)
                    keep_min_tagged(vmax(a[m], n[q]), bv[q]);
                else
                    keep_min(vmax(a[m], n[q]), uint32_t(it) << 8 | m, bv[q], bi[q]);
            }
            a[m] += V(1);
        }
    }
    unsigned long long acc = 0;
#pragma unroll
    for (int q = 0; q < kAcc; q++) acc += (unsigned long long)bv[q] + bi[q];
    if (acc == 0x123456789ull) *sink = acc;   // keeps the work alive
}

}  // namespace

// Measured relaxations per second (one relaxation = one candidate against one cell)
// of the plain 32-bit (wide = 0), 64-bit (wide = 1) or tagged 32-bit (wide = 2) word
// arithmetic on every SM of the current device.  Returns 0 on success, -1 on a CUDA
// error or an unknown mode.
extern "C" int nest_peak_relax(int wide, int iters, double *relax_per_s) {
    if (wide < 0 || wide > 2) return -1;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
        return -1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, wide == 1 ? peak_kernel<uint64_t, false> : wide == 2 ? peak_kernel<uint32_t, true> : peak_kernel<uint32_t, false>,
        kThreads, 0);
    if (per_sm < 1) per_sm = 1;
    unsigned long long *sink = nullptr;
    if (cudaMalloc(&sink, sizeof *sink) != cudaSuccess) return -1;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    const dim3 grid(unsigned(sms * per_sm));
    for (int rep = 0; rep < 2; rep++) {   // the first launch warms up
        cudaEventRecord(e0);
        if (wide == 1)
            peak_kernel<uint64_t, false><<<grid, kThreads>>>(iters, 12345u, sink);
        else if (wide == 2)
            peak_kernel<uint32_t, true><<<grid, kThreads>>>(iters, 12345u, sink);
        else
            peak_kernel<uint32_t, false><<<grid, kThreads>>>(iters, 12345u, sink);
        cudaEventRecord(e1);
    }
    float ms = 0;
    const bool ok = cudaEventSynchronize(e1) == cudaSuccess && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(sink);
    if (!ok || ms <= 0) return -1;
    *relax_per_s = double(grid.x) * kThreads * double(iters) * kCand * kAcc / (ms * 1e-3);
    return 0;
}
