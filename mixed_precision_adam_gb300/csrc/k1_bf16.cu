// k1_bf16.cu -- K1 reduce/prepare kernels for bf16 replica grads (one grad
// dtype per translation unit, so the three compile in parallel).
#include "k1.cuh"

namespace dopt {

int launch_k1_bf16(K1Params& kp, const K1Launch& l, cudaStream_t s) { return launch_k1_for<__nv_bfloat16>(kp, l, s); }

}  // namespace dopt
