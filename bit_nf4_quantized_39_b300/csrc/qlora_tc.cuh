// qlora_tc.cuh -- tensor-core (tcgen05) fused layer kernels.  Placeholder
// interface: the tcgen05 path is not enabled in this build yet, so every
// shape takes the CUDA-core kernels.
#pragma once

#include "common.cuh"

namespace qn {

inline size_t tc_ws_bytes(int64_t, int64_t, int64_t, int32_t) { return 0; }
inline bool tc_supported(int64_t, int64_t, int64_t, int32_t) { return false; }
inline bool tc_bwd_supported(int64_t, int64_t, int64_t, int32_t) { return false; }
template <typename SpanT>
inline int launch_tc_fwd(const QnNF4View &, const uint16_t *, int64_t, const float *, const uint16_t *, int,
                         uint16_t *, SpanT &, cudaStream_t) { return -1; }
template <typename SpanT>
inline int launch_tc_bwd(const QnNF4View &, const uint16_t *, int64_t, const float *, const uint16_t *, int,
                         uint16_t *, SpanT &, cudaStream_t) { return -1; }

}  // namespace qn
