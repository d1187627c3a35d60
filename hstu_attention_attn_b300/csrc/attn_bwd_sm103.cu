// attn_bwd_sm103.cu -- jagged HSTU attention backward on tcgen05 (in progress).
#include "common.cuh"
#include "plan.cuh"

namespace mtgr {

cudaError_t launch_attn_bwd_bf16(const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*, int64_t,
                                 const __nv_bfloat16*, int64_t, int, int, const int32_t*, int32_t, const int64_t*,
                                 float*, __nv_bfloat16*, __nv_bfloat16*, __nv_bfloat16*, int64_t,
                                 const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*, int32_t*,
                                 cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mtgr
