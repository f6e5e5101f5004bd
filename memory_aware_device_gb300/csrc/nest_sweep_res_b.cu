// Resident DP sweep instantiated for 3 and 4 link candidates (the kernels are in
// nest_sweep.cuh); a translation unit of its own so that the instantiations compile in
// parallel.
#include "nest_sweep.cuh"

namespace nest {

int resident_capacity_34(int CT, int KT, int cluster, int threads, size_t smem) {
    if (CT == 3) return resident_capacity_kt<3>(KT, cluster, threads, smem);
    return resident_capacity_kt<4>(KT, cluster, threads, smem);
}

int launch_resident_34(int CT, const PassArgs &a, void *stream) {
    if (CT == 3) return launch_resident_kt<3>(a, stream);
    return launch_resident_kt<4>(a, stream);
}

}  // namespace nest
