// Decode attention over keys cached before the rotary position embedding
// (kvq_decode_attention_rope): launcher shared by the ABI and the kernel unit.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

// Query heads per KV head the kernel is built for.
inline bool rope_group_supported(int rg) { return rg == 1 || rg == 2 || rg == 4; }

// Positions must be exact in fp32.
constexpr int64_t kRopeMaxPositions = 1LL << 24;

// ws: the decode workspace (kvq_workspace_bytes, zero-filled; left zero).
cudaError_t launch_decode_rope(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                               int64_t n_resid, int64_t n_sink, int64_t ring_head,
                               const __half *q, float *out, float scale, double rope_base,
                               void *ws, int num_sms, cudaStream_t st);

}  // namespace kvq
