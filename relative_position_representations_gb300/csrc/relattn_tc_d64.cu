// tcgen05 path, head dimension 64.
#include "relattn_tc_launch.cuh"

namespace relattn {
cudaError_t launch_tc_bf16_d64(const TcArgs &a, const T5Buckets *t5, int *err, cudaStream_t s) {
    return tc::launch_tc<64>(a, t5, err, s);
}
}  // namespace relattn
