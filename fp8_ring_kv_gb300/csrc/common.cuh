// Internal definitions shared by the kvring kernels and the host launcher.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace kvring_dev {

constexpr int kMaxAxes = 3;
constexpr float kE4m3Max = 448.0f;

// state words at the start of the workspace
// ST_STATIC: 1 once a ring with per-head fixed scales has been calibrated
enum : int { ST_WP = 0, ST_NVALID = 1, ST_ERR = 2, ST_DONE = 3, ST_STATIC = 4, ST_WORDS = 64 };
// per-head fixed scales, fp32 [6][H]: the recorded maxima of K and V, then
// (scale, inv) of K and of V
enum : int { STAT_AMAX_K = 0, STAT_AMAX_V = 1, STAT_K_SCALE = 2, STAT_K_INV = 3, STAT_V_SCALE = 4, STAT_V_INV = 5 };
enum : int { DEVERR_POS_RANGE = 1, DEVERR_EMPTY = 2, DEVERR_TIMEOUT = 4 };

// Device view of one ring, passed by value to every kernel.
struct RingView {
  int32_t* state;                 // ST_* words
  const float2* rope[kMaxAxes];   // per axis: [pos_count][axis_dims/2] (cos, sin)
  int32_t pos_min[kMaxAxes];
  int32_t pos_count[kMaxAxes];
  int32_t axis_pairs[kMaxAxes];   // axis_dims / 2
  int32_t pair_off[kMaxAxes];     // index of the first pair of each axis
  uint8_t* k_codes;               // [H][S][D]
  uint8_t* v_codes;               // [H][S][D]
  float* k_scale;                 // [H][S_pad]
  float* v_scale;                 // [H][S_pad]
  uint8_t* q_codes;               // query scratch: e4m3 [n_q][H][D]
  float* q_scale;                 // query scratch: fp32 [H][Q_pad]
  int32_t H, D, S, S_pad, n_axes, Q_pad;
  int32_t G;                      // global slots 0 .. G-1; the window ring is slots G .. S-1
  float* stat;                    // per-head fixed scales [6][H] (STAT_*)
  int32_t scale_mode;             // 0: per (token, head) scales; 1: per head, fixed by calibration
  const uint4* gamma_k;           // RMS-norm weights of K, bf16 [H][D] (null: no norm)
  const uint4* gamma_q;           // RMS-norm weights of Q, bf16 [H][D] (null: no norm)
  float norm_eps;
  float* head_stat;               // query scratch: fp32 [H][2] per call: (c, floor) of the attention, below
};

// ---------------------------------------------------------------- attention range factors
// The attention stores weights P = e * w * 2^c in fp16 with e <= 2^kAttnLazyLog2
// and w = max(s_v, floor) per slot; per head, from the largest V scale m over
// the valid slots: c = 14 - kAttnLazyLog2 - floor(log2 m) (0 if m = 0, clamped
// to [-64, 64]) keeps every P below 2^15, and floor = 2^-kAttnFloorLog2 *
// max(m, 2^-c) keeps 2^-c / w <= 2^kAttnFloorLog2 inside fp16.
constexpr int kAttnLazyLog2 = 10;
constexpr int kAttnFloorLog2 = 15;

__device__ __forceinline__ void attn_head_factors(float max_sv, float& c, float& floor) {
  int ci = max_sv > 0.0f ? 14 - kAttnLazyLog2 - ilogbf(max_sv) : 0;
  ci = ci < -64 ? -64 : (ci > 64 ? 64 : ci);
  c = (float)ci;
  floor = ldexpf(fmaxf(max_sv, ldexpf(1.0f, -ci)), -kAttnFloorLog2);
}

// ---------------------------------------------------------------- numerics
// These are the exact fp32 operation sequences the method fixes; the compiler
// must not contract or reorder them (no fast-math, explicit _rn intrinsics).

// One RoPE pair: (x0 c - x1 s, x0 s + x1 c), every product and sum rounded
// (the _rn intrinsics are never contracted into a fused multiply-add).
__device__ __forceinline__ void rope_pair(float& x0, float& x1, float c, float s) {
  const float a = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
  const float b = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
  x0 = a;
  x1 = b;
}

// Scale and its inverse for a row whose absolute maximum is ``amax``:
// scale = amax / 448, inv = 448 / amax, both IEEE-rounded; zero rows get 0.
__device__ __forceinline__ void absmax_scale(float amax, float& scale, float& inv) {
  if (amax > 0.0f) {
    scale = __fdiv_rn(amax, kE4m3Max);
    inv = __fdiv_rn(kE4m3Max, amax);
  } else {
    scale = 0.0f;
    inv = 0.0f;
  }
}

// The same scale and inverse for a row of D = 16 L channels held by L lanes
// (mask gm): each lane makes one of the two divisions -- the row's first
// lane amax / 448, its second 448 / amax -- and the row shares them.  Bit for
// bit the values of absmax_scale.
template <int L>
__device__ __forceinline__ void row_absmax_scale(float amax, float& scale, float& inv, unsigned gm) {
  if constexpr (L == 1) {
    absmax_scale(amax, scale, inv);
  } else {
    const int lane = threadIdx.x & 31;
    const int base = lane & ~(L - 1);
    const bool first = (lane & (L - 1)) == 0;
    const float q = amax > 0.0f ? __fdiv_rn(first ? amax : kE4m3Max, first ? kE4m3Max : amax) : 0.0f;
    scale = __shfl_sync(gm, q, base);
    inv = __shfl_sync(gm, q, base + 1);
  }
}

// 16 values -> 16 e4m3 codes (round to nearest even, saturating) of x * inv.
// A zero row (inv == 0) gives all-zero codes (+0).
__device__ __forceinline__ uint4 quant16(const float* x, float inv) {
  uint32_t w[4];
  const float2 iv = make_float2(inv, inv);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = __fmul2_rn(make_float2(x[4 * i + 0], x[4 * i + 1]), iv);
    const float2 b = __fmul2_rn(make_float2(x[4 * i + 2], x[4 * i + 3]), iv);
    const uint32_t lo = cvt_e4m3x2(a.x, a.y);
    const uint32_t hi = cvt_e4m3x2(b.x, b.y);
    w[i] = lo | (hi << 16);
  }
  if (inv == 0.0f) w[0] = w[1] = w[2] = w[3] = 0u;
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// 16 e4m3 codes -> 16 fp32 values (exact).
__device__ __forceinline__ void dequant16_codes(uint4 c, float* x) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = cvt_e4m3x2_to_f16x2((uint16_t)(w[i] & 0xFFFFu));
    const uint32_t hi = cvt_e4m3x2_to_f16x2((uint16_t)(w[i] >> 16));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    x[4 * i + 0] = a.x;
    x[4 * i + 1] = a.y;
    x[4 * i + 2] = b.x;
    x[4 * i + 3] = b.y;
  }
}

// 16 e4m3 codes -> 16 fp32 values code * scale, each product rounded once.
__device__ __forceinline__ void dequant16_scaled(uint4 c, float scale, float* x) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  const float2 sc = make_float2(scale, scale);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = cvt_e4m3x2_to_f16x2((uint16_t)(w[i] & 0xFFFFu));
    const uint32_t hi = cvt_e4m3x2_to_f16x2((uint16_t)(w[i] >> 16));
    const float2 a = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&lo)), sc);
    const float2 b = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&hi)), sc);
    x[4 * i + 0] = a.x;
    x[4 * i + 1] = a.y;
    x[4 * i + 2] = b.x;
    x[4 * i + 3] = b.y;
  }
}

// 8 bf16 (one uint4) -> 8 fp32 (exact).
__device__ __forceinline__ void bf16x8_to_f32(uint4 u, float* x) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i + 0] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// RMS norm of one row of D = 16 L channels held as 16 per lane (L lanes of
// one warp, mask gm), in place: S = sum x^2 in fp64 (exact for bf16 inputs
// unless a row spans an extreme dynamic range), rounded once to fp32;
// ms = S / D (exact); rstd = 1/sqrt(ms + eps), correctly rounded; then
// x = bf16(fl32(fl32(x * rstd) * gamma)).  g: this lane's 16 weights.
template <int L>
__device__ __forceinline__ void rms_norm16(float* x, const uint4* g, float eps, unsigned gm) {
  double s = 0.0;
#pragma unroll
  for (int i = 0; i < 16; ++i) s += (double)x[i] * (double)x[i];
#pragma unroll
  for (int off = L / 2; off > 0; off >>= 1) s += __shfl_xor_sync(gm, s, off);
  const float ms = __fmul_rn(__double2float_rn(s), 1.0f / (float)(16 * L));
  const float rstd = __frsqrt_rn(__fadd_rn(ms, eps));
  float w[16];
  bf16x8_to_f32(__ldg(g), w);
  bf16x8_to_f32(__ldg(g + 1), w + 8);
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(x[i], rstd), w[i])));
}

// The axis and in-axis index of RoPE pair p, and its table entry for the
// given positions.  Out-of-range positions are clamped and flagged.
__device__ __forceinline__ float2 rope_cs(const RingView& rv, const int32_t* pos_row, int p, bool& bad) {
  int a = 0;
  if (rv.n_axes > 1 && p >= rv.pair_off[1]) a = 1;
  if (rv.n_axes > 2 && p >= rv.pair_off[2]) a = 2;
  const int j = p - rv.pair_off[a];
  int idx = pos_row[a] - rv.pos_min[a];
  if (idx < 0 || idx >= rv.pos_count[a]) {
    bad = true;
    idx = idx < 0 ? 0 : rv.pos_count[a] - 1;
  }
  return __ldg(rv.rope[a] + (size_t)idx * rv.axis_pairs[a] + j);
}

}  // namespace kvring_dev
