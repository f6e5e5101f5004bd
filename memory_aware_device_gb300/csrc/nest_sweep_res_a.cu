// Resident DP sweep instantiated for 1 and 2 link candidates (the kernels are in
// nest_sweep.cuh); a translation unit of its own so that the instantiations compile in
// parallel.
#include "nest_sweep.cuh"

namespace nest {

int resident_capacity_12(int CT, int KT, int cluster, int threads, size_t smem) {
    if (CT == 1) return resident_capacity_kt<1>(KT, cluster, threads, smem);
    return resident_capacity_kt<2>(KT, cluster, threads, smem);
}

int launch_resident_12(int CT, const PassArgs &a, void *stream) {
    if (CT == 1) return launch_resident_kt<1>(a, stream);
    return launch_resident_kt<2>(a, stream);
}

}  // namespace nest
