// tcgen05 path, head dimension 128.
#include "relattn_tc_launch.cuh"

namespace relattn {
cudaError_t launch_tc_bf16_d128(const TcArgs &a, const T5Buckets *t5, int *err, cudaStream_t s) {
    return tc::launch_tc<128>(a, t5, err, s);
}
}  // namespace relattn
