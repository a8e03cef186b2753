// Decode attention over keys cached before the rotary position embedding
// (kvq_decode_attention_rope): launcher shared by the ABI and the kernel unit.
#pragma once

#include <math.h>

#include "kvq_internal.cuh"

namespace kvq {

// Query heads per KV head the kernel is built for.
inline bool rope_group_supported(int rg) { return rg == 1 || rg == 2 || rg == 4; }

// Positions must be exact in fp32.
constexpr int64_t kRopeMaxPositions = 1LL << 24;

// cos and sin of delta * theta for a non-negative integer delta below 2^24:
// the product as a float-float (theta = th.x + th.y), reduced by 2 pi given in
// three parts c1 + c2 + c3 (W. J. Cody, W. Waite, "Software Manual for the
// Elementary Functions", 1980), then __sincosf of the reduced angle.  Returns
// (cos, sin).
__device__ __forceinline__ float2 rope_cos_sin(float delta, float2 th, float c1, float c2,
                                               float c3) {
  const float p = __fmul_rn(delta, th.x);
  const float e = fmaf(delta, th.x, -p) + delta * th.y;  // p + e = delta * theta
  const float k = rintf(p * 0.15915494309189535f);
  float r = fmaf(-k, c1, p);
  r = fmaf(-k, c2, r);
  r = fmaf(-k, c3, r);
  r += e;
  float s, c;
  __sincosf(r, &s, &c);
  return make_float2(c, s);
}

// theta_i = base^(-2i/d) as float hi + lo, and 2 pi as c1 + c2 + c3.
inline void rope_constants(double base, int d, float2 *theta, float &c1, float &c2, float &c3) {
  for (int i = 0; i < d / 2; ++i) {
    const double th = pow(base, -2.0 * i / d);
    const float hi = (float)th;
    theta[i] = make_float2(hi, (float)(th - (double)hi));
  }
  const double two_pi = 2.0 * M_PI;
  c1 = (float)two_pi;
  c2 = (float)(two_pi - (double)c1);
  c3 = (float)(two_pi - (double)c1 - (double)c2);
}

// The tensor-core form (head_dim 128, one query head per KV head, KIVI with
// key groups of 32 or more, fp32 statistics, no cache options): true when
// launch_decode_tc_rope takes the call.
bool tc_rope_supported(const Geometry &g);
int tc_rope_variant_name(const Geometry &g, char *buf, size_t len);

// ws: as launch_decode_rope.  Positions: token i of the cache sits at i, the
// query at n_quant + n_resid - 1.
cudaError_t launch_decode_tc_rope(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                                  int64_t n_resid, const __half *q, float *out, float scale,
                                  double rope_base, void *ws, int num_sms, cudaStream_t st);

// ws: the decode workspace (kvq_workspace_bytes, zero-filled; left zero).
cudaError_t launch_decode_rope(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                               int64_t n_resid, int64_t n_sink, int64_t ring_head,
                               const __half *q, float *out, float scale, double rope_base,
                               void *ws, int num_sms, cudaStream_t st);

}  // namespace kvq
