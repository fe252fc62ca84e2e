// tcgen05 (sm_103a) kernels: declarations of the fast-path dispatch.  The kernels follow.
#pragma once

#include "sched.cuh"
#include "simt_attention.cuh"

namespace mla {

inline bool tc_attention_supported(const mla_config*, const mla_cache*, int, int) { return false; }
inline mla_status tc_attention_launch(const AttnArgs&, const mla_cache*, unsigned long long, cudaStream_t) {
    return MLA_ERR_UNSUPPORTED;
}
inline bool tc_gemm_append_supported(const mla_config*, int) { return false; }
inline mla_status tc_gemm_append(const mla_config*, const mla_cache*, const void*, const void*, const void*,
                                 const int32_t*, const int32_t*, int32_t, cudaStream_t) {
    return MLA_ERR_UNSUPPORTED;
}
inline bool tc_gemm_absorb_supported(const mla_config*, int) { return false; }
inline mla_status tc_gemm_absorb(const mla_config*, const void*, const void*, void*, int32_t, cudaStream_t) {
    return MLA_ERR_UNSUPPORTED;
}
inline bool tc_gemm_out_supported(const mla_config*, int) { return false; }
inline mla_status tc_gemm_out(const mla_config*, const void*, const void*, void*, int32_t, cudaStream_t) {
    return MLA_ERR_UNSUPPORTED;
}

}  // namespace mla
