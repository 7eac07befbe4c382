// fp8_ring_attn: n_q bf16 queries attend over every valid slot of the FP8 ring.
//
// Runway Characters paper, §4.3 (K and V stored as float8_e4m3, the queries
// quantised per call, attention reading the FP8 cache directly) and
// Appendix G (each call reads all the cache's slots; no causal mask).
//
// One block per (tile of 128 queries, head).  The slots are visited in tiles
// of 128 in storage order: attention is a sum over the valid slots, so the
// ring's wrap needs no reordering, and slots >= n_valid are masked.
//
//   S_j  = Qcodes . Kcodes_j^T            tcgen05 kind::f8f6f4, fp32 in TMEM
//   t    = S_j * s_k (per column);  logit*log2(e) = t * s_q * log2(e)/sqrt(D)
//   online softmax in base 2: e = exp2(t*r - m + c), l += e, with a running
//   row maximum m that is only raised (and O rescaled) when a tile's maximum
//   exceeds it by more than 2^8, so e <= 2^8 * 2^c
//   P    = e * s_v (per column) rounded to fp16, stored to TMEM
//   O   += P . Vcodes_j                    tcgen05 kind::f16 (A = P from TMEM)
//   out  = O / l
// The e4m3 V codes are widened to fp16 in shared memory (exact) because the
// fp16 MMA takes both operands in fp16; P in fp16 keeps the weighted sum of V
// within the accuracy that e4m3 weights would lose.  2^c is a per-head power of
// two (cancelling between O and l) that keeps P within fp16 range.
//
// Warp roles (320 threads):
//   warps 0-3  softmax + epilogue, thread r owns query row r (TMEM lane r)
//   warps 4-7  prologue (RoPE + e4m3 of the 128 query rows, C_v), then the
//              per-tile widening of V to fp16
//   warp 8     TMA producer (K, V codes and their scales, 2 stages)
//   warp 9     TMEM allocation and MMA issue
#include <cfloat>

#include "common.cuh"
#include "launch.h"

namespace kvring_dev {

constexpr int BM = 128;           // query rows per block
constexpr int BN = 128;           // slots per tile
constexpr int NSTAGE = 2;         // fp8 K/V stages
constexpr int ATT_THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;      // two fp32 S buffers at columns 0 and 128
constexpr uint32_t TM_P = 256;    // two fp16 P buffers (64 columns each) at 256 and 320
constexpr uint32_t TM_O = 384;    // fp32 O accumulator (D columns)
constexpr float kLazyRescale = 8.0f;   // log2 of the largest unnormalised weight

template <int D>
struct AttnLayout {
  static constexpr int Q = 0;                            // e4m3 [BM][D], K-major swizzled
  static constexpr int K0 = Q + BM * D;                  // NSTAGE x e4m3 [BN][D]
  static constexpr int V0 = K0 + NSTAGE * BN * D;        // NSTAGE x e4m3 [BN][D]
  static constexpr int VH0 = V0 + NSTAGE * BN * D;       // 2 x fp16 [BN][D], MN-major swizzled
  static constexpr int SK0 = VH0 + 2 * BN * D * 2;       // NSTAGE x fp32 [BN]
  static constexpr int SV0 = SK0 + NSTAGE * BN * 4;
  static constexpr int SQ = SV0 + NSTAGE * BN * 4;       // fp32 [BM]
  static constexpr int BAR = SQ + BM * 4;
  static constexpr int NBAR = 16;
  static constexpr int MISC = BAR + NBAR * 8;
  static constexpr int BYTES = MISC + 64;
  static constexpr int ALLOC = BYTES + 1024;             // slack for 1024-byte alignment
};

// byte offset of 16-byte chunk c of row r in a K-major tile whose rows are
// D bytes (D = 128: 128-byte swizzle; D = 64: 64-byte swizzle)
template <int D>
__device__ __forceinline__ int kmajor_chunk(int r, int c) {
  if constexpr (D == 128)
    return r * 128 + ((c ^ (r & 7)) << 4);
  else
    return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

template <int D>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t addr) {
  if constexpr (D == 128)
    return make_sdesc_sw128(addr, 16, 1024);
  else
    return make_sdesc_sw64(addr, 16, 512);
}

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    fp8_ring_attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmSK, const __grid_constant__ CUtensorMap tmSV,
                         RingView rv, const uint4* __restrict__ q, const int32_t* __restrict__ q_pos, int n_q,
                         void* __restrict__ out, int out_f32) {
  using LY = AttnLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LY::BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 2;
  uint64_t* s_full = bars + 4;
  uint64_t* s_empty = bars + 6;
  uint64_t* vh_full = bars + 8;
  uint64_t* p_full = bars + 10;
  uint64_t* pv_done = bars + 12;
  uint64_t* q_full = bars + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LY::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY::MISC + 4);
  int* maxsv_bits = reinterpret_cast<int*>(sm + LY::MISC + 8);
  float* cv_smem = reinterpret_cast<float*>(sm + LY::MISC + 12);   // log2 of the per-head weight factor
  float* sq_smem = reinterpret_cast<float*>(sm + LY::SQ);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int qt = blockIdx.x;
  const int h = blockIdx.y;
  const int H = rv.H;
  const int n_valid = rv.state[ST_NVALID];
  const int T = (n_valid + BN - 1) / BN;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1 + 4 + 4);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
      mbar_init(&vh_full[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(q_full, 4);
    *abort_flag = 0;
    *maxsv_bits = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmSK);
    tma_prefetch_desc(&tmSV);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (n_valid <= 0) {
    // nothing to attend to: zeros, and a flag the host can read
    if (warp < 4) {
      const int qi = qt * BM + tid;
      if (qi < n_q) {
        const int bytes = D * (out_f32 ? 4 : 2);
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + ((size_t)qi * H + h) * bytes);
        for (int i = 0; i < bytes / 16; ++i) o[i] = make_uint4(0, 0, 0, 0);
      }
    }
    if (tid == 0 && qt == 0 && h == 0) atomicOr(&rv.state[ST_ERR], DEVERR_EMPTY);
  } else if (warp < 4) {
    // ======================================================== softmax + epilogue
    const int r = tid;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    constexpr float kRowC = (D == 128 ? 0.08838834764831845f : 0.125f) * 1.4426950408889634f;
    bool ok = mbar_wait(q_full, 0, abort_flag);
    const float sq = sq_smem[r];
    const float rq = sq > 0.0f ? sq * kRowC : 1.0f;
    const float log2cv = *cv_smem;
    float m_run = -INFINITY;
    float2 lacc = make_float2(0.0f, 0.0f);
    for (int j = 0; ok && j < T; ++j) {
      const int s = j % NSTAGE;
      const int b = j & 1;
      if (!mbar_wait(&kv_full[s], (j / NSTAGE) & 1, abort_flag) || !mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4* sk4 = reinterpret_cast<const float4*>(sm + LY::SK0 + s * BN * 4);
      const float4* sv4 = reinterpret_cast<const float4*>(sm + LY::SV0 + s * BN * 4);
      const int valid = min(BN, n_valid - j * BN);
      const uint32_t s_addr = tmem + lane_off + TM_S + b * 128;

      // pass 1: the tile's row maximum of t = S * s_k
      float mt = -INFINITY;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t x[32];
        tmem_ld32(s_addr + cb * 32, x);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 k4 = sk4[(cb * 32 + i) >> 2];
          float2 t0 = mul2(make_float2(__uint_as_float(x[i]), __uint_as_float(x[i + 1])), make_float2(k4.x, k4.y));
          float2 t1 = mul2(make_float2(__uint_as_float(x[i + 2]), __uint_as_float(x[i + 3])), make_float2(k4.z, k4.w));
          if (valid < BN) {
            const int c = cb * 32 + i;
            if (c >= valid) t0.x = -INFINITY;
            if (c + 1 >= valid) t0.y = -INFINITY;
            if (c + 2 >= valid) t1.x = -INFINITY;
            if (c + 3 >= valid) t1.y = -INFINITY;
          }
          mt = max3f(mt, t0.x, t0.y);
          mt = max3f(mt, t1.x, t1.y);
        }
      }
      // raise the running maximum only when it is exceeded by more than 2^8
      const float m_tile = mt * rq;
      const bool grow = (j == 0) || (m_tile > m_run + kLazyRescale);
      if (__any_sync(0xFFFFFFFFu, grow)) {
        const float m_new = fmaxf(m_run, m_tile);
        if (j > 0) {
          // O holds rows weighted by exp2(-m_run): bring them to exp2(-m_new)
          if (!mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = ex2f(m_run - m_new);
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t o[16];
            tmem_ld16(tmem + lane_off + TM_O + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(tmem + lane_off + TM_O + c0, o);
          }
          tmem_wait_st();
          lacc.x *= alpha;
          lacc.y *= alpha;
        }
        m_run = m_new;
      }
      // P buffer b is free once PV of tile j-2 has finished
      if (j >= 2 && !mbar_wait(&pv_done[b], ((j - 2) >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // pass 2: e = exp2(t*r - m + c), l += e, P = e * s_v -> fp16 -> TMEM
      const float2 rq2 = make_float2(rq, rq);
      const float2 moff = make_float2(log2cv - m_run, log2cv - m_run);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t x[32];
        tmem_ld32(s_addr + cb * 32, x);
        tmem_wait_ld();
        if (cb == 3) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[b]);
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 k4 = sk4[(cb * 32 + i) >> 2];
          const float4 v4 = sv4[(cb * 32 + i) >> 2];
          float2 t0 = mul2(make_float2(__uint_as_float(x[i]), __uint_as_float(x[i + 1])), make_float2(k4.x, k4.y));
          float2 t1 = mul2(make_float2(__uint_as_float(x[i + 2]), __uint_as_float(x[i + 3])), make_float2(k4.z, k4.w));
          t0 = fma2(t0, rq2, moff);
          t1 = fma2(t1, rq2, moff);
          float2 e0 = make_float2(ex2f(t0.x), ex2f(t0.y));
          float2 e1 = make_float2(ex2f(t1.x), ex2f(t1.y));
          if (valid < BN) {
            const int c = cb * 32 + i;
            if (c >= valid) e0.x = 0.0f;
            if (c + 1 >= valid) e0.y = 0.0f;
            if (c + 2 >= valid) e1.x = 0.0f;
            if (c + 3 >= valid) e1.y = 0.0f;
          }
          lacc = add2(lacc, add2(e0, e1));
          const float2 p0 = mul2(e0, make_float2(v4.x, v4.y));
          const float2 p1 = mul2(e1, make_float2(v4.z, v4.w));
          pk[i >> 1] = cvt_f16x2(p0.x, p0.y);
          pk[(i >> 1) + 1] = cvt_f16x2(p1.x, p1.y);
        }
        tmem_st16(tmem + lane_off + TM_P + b * 64 + cb * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_full[b]);
        mbar_arrive(&kv_empty[s]);
      }
    }
    const float l_run = lacc.x + lacc.y;
    // epilogue: out = O / l
    if (ok && mbar_wait(&pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, abort_flag)) {
      tc_fence_after();
      const int qi = qt * BM + r;
      const float scale = 1.0f / l_run;
      uint8_t* orow = static_cast<uint8_t*>(out) + ((size_t)qi * H + h) * (size_t)D * (out_f32 ? 4 : 2);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        uint32_t o[16];
        tmem_ld16(tmem + lane_off + TM_O + c0, o);
        tmem_wait_ld();
        if (qi < n_q) {
          if (out_f32) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 4);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(__float_as_uint(__uint_as_float(o[4 * i]) * scale),
                                  __float_as_uint(__uint_as_float(o[4 * i + 1]) * scale),
                                  __float_as_uint(__uint_as_float(o[4 * i + 2]) * scale),
                                  __float_as_uint(__uint_as_float(o[4 * i + 3]) * scale));
          } else {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const __nv_bfloat162 v2 =
                  __floats2bfloat162_rn(__uint_as_float(o[2 * i]) * scale, __uint_as_float(o[2 * i + 1]) * scale);
              pk[i] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 2);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
    }
    tc_fence_before();
  } else if (warp < 8) {
    // ======================================================== prologue + V widening
    const int ct = tid - 128;
    // C_v from the largest V scale of this head
    float mx = 0.0f;
    const float* vs = rv.v_scale + (size_t)h * rv.S_pad;
    for (int i = ct; i < n_valid; i += 128) mx = fmaxf(mx, vs[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    if (lane == 0) atomicMax(maxsv_bits, __float_as_int(mx));

    // query row ct: RoPE in fp32, e4m3 with its own absmax scale
    const int qi = qt * BM + ct;
    uint8_t* qtile = sm + LY::Q;
    float sq = 0.0f;
    bool bad = false;
    if (qi < n_q) {
      float x[D];
      const uint4* src = q + ((size_t)qi * H + h) * (D / 8);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) bf16x8_to_f32(__ldg(src + i), x + 8 * i);
      const int32_t* pr = q_pos + (size_t)qi * rv.n_axes;
#pragma unroll
      for (int p = 0; p < D / 2; ++p) {
        const float2 cs = rope_cs(rv, pr, p, bad);
        rope_pair(x[2 * p], x[2 * p + 1], cs.x, cs.y);
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < D; ++i) amax = fmaxf(amax, fabsf(x[i]));
      float inv;
      absmax_scale(amax, sq, inv);
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        *reinterpret_cast<uint4*>(qtile + kmajor_chunk<D>(ct, c)) = quant16(x + 16 * c, inv);
    } else {
#pragma unroll
      for (int c = 0; c < D / 16; ++c) *reinterpret_cast<uint4*>(qtile + kmajor_chunk<D>(ct, c)) = make_uint4(0, 0, 0, 0);
    }
    sq_smem[ct] = sq;
    if (bad) atomicOr(&rv.state[ST_ERR], DEVERR_POS_RANGE);
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (ct == 0) {
      const float m = __int_as_float(*maxsv_bits);
      // weights reach 2^8 * 2^c; with c = 6 - floor(log2 max s_v) every
      // P = weight * s_v stays below 2^15 (fp16 max 65504)
      int c = m > 0.0f ? 6 - ilogbf(m) : 0;
      c = c < -64 ? -64 : (c > 64 ? 64 : c);
      *cv_smem = (float)c;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);

    constexpr int CH = D / 16;  // 16-byte e4m3 chunks per slot row
    for (int j = 0; j < T; ++j) {
      const int s = j % NSTAGE;
      const int b = j & 1;
      if (!mbar_wait(&kv_full[s], (j / NSTAGE) & 1, abort_flag)) break;
      if (j >= 2 && !mbar_wait(&pv_done[b], ((j - 2) >> 1) & 1, abort_flag)) break;
      const uint8_t* vsrc = sm + LY::V0 + s * BN * D;
      uint8_t* vdst = sm + LY::VH0 + b * BN * D * 2;
      // eight consecutive threads take the same chunk of eight consecutive
      // slots, so their 16-byte reads and writes fall in distinct bank groups
#pragma unroll
      for (int it = 0; it < BN * CH / 128; ++it) {
        const int task = it * 128 + ct;
        const int sl = 8 * (task / (8 * CH)) + (task & 7);
        const int c = (task >> 3) % CH;
        const uint4 u = *reinterpret_cast<const uint4*>(vsrc + kmajor_chunk<D>(sl, c));
        uint4 o0, o1;
        o0.x = cvt_e4m3x2_to_f16x2((uint16_t)(u.x & 0xFFFFu));
        o0.y = cvt_e4m3x2_to_f16x2((uint16_t)(u.x >> 16));
        o0.z = cvt_e4m3x2_to_f16x2((uint16_t)(u.y & 0xFFFFu));
        o0.w = cvt_e4m3x2_to_f16x2((uint16_t)(u.y >> 16));
        o1.x = cvt_e4m3x2_to_f16x2((uint16_t)(u.z & 0xFFFFu));
        o1.y = cvt_e4m3x2_to_f16x2((uint16_t)(u.z >> 16));
        o1.z = cvt_e4m3x2_to_f16x2((uint16_t)(u.w & 0xFFFFu));
        o1.w = cvt_e4m3x2_to_f16x2((uint16_t)(u.w >> 16));
        // channels 16c .. 16c+15 -> MN-major fp16 tile: 64-channel column
        // blocks of [BN][128 bytes], 128-byte swizzle by slot
        const int d0 = 16 * c;
        uint8_t* base = vdst + (d0 >> 6) * (BN * 128) + sl * 128;
        const int cc = (d0 & 63) >> 3;
        *reinterpret_cast<uint4*>(base + ((cc ^ (sl & 7)) << 4)) = o0;
        *reinterpret_cast<uint4*>(base + (((cc + 1) ^ (sl & 7)) << 4)) = o1;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&vh_full[b]);
        mbar_arrive(&kv_empty[s]);
      }
    }
  } else if (warp == 8) {
    // ======================================================== TMA producer
    if (lane == 0) {
      for (int j = 0; j < T; ++j) {
        const int s = j % NSTAGE;
        if (j >= NSTAGE && !mbar_wait(&kv_empty[s], ((j / NSTAGE) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(&kv_full[s], 2 * BN * D + 2 * BN * 4);
        tma_load_3d(sm + LY::K0 + s * BN * D, &tmK, &kv_full[s], 0, j * BN, h);
        tma_load_3d(sm + LY::V0 + s * BN * D, &tmV, &kv_full[s], 0, j * BN, h);
        tma_load_2d(sm + LY::SK0 + s * BN * 4, &tmSK, &kv_full[s], j * BN, h);
        tma_load_2d(sm + LY::SV0 + s * BN * 4, &tmSV, &kv_full[s], j * BN, h);
      }
    }
  } else {
    // ======================================================== MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc(0, 0, 0, 0, BM, BN);   // e4m3 x e4m3, both K-major
      constexpr uint32_t idesc_pv = make_idesc(0, 0, 0, 1, BM, D);    // f16 x f16, V MN-major
      bool ok = mbar_wait(q_full, 0, abort_flag);
      const uint32_t q_addr = smem_u32(sm + LY::Q);
      auto issue_pv = [&](int i) -> bool {
        const int b = i & 1;
        if (!mbar_wait(&p_full[b], (i >> 1) & 1, abort_flag) || !mbar_wait(&vh_full[b], (i >> 1) & 1, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t va = smem_u32(sm + LY::VH0 + b * BN * D * 2);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_f16_ts(tmem + TM_O, tmem + TM_P + b * 64 + kk * 8, make_sdesc_sw128(va + kk * 16 * 128, BN * 128, 1024),
                     idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&pv_done[b]);
        return true;
      };
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % NSTAGE;
        const int b = j & 1;
        if (!mbar_wait(&kv_full[s], (j / NSTAGE) & 1, abort_flag) ||
            (j >= 2 && !mbar_wait(&s_empty[b], ((j >> 1) - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ka = smem_u32(sm + LY::K0 + s * BN * D);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          mma_f8_ss(tmem + TM_S + b * 128, kmajor_desc<D>(q_addr + kk * 32), kmajor_desc<D>(ka + kk * 32), idesc_qk,
                    kk > 0 ? 1u : 0u);
        mma_commit(&s_full[b]);
        mma_commit(&kv_empty[s]);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(T - 1);
    }
  }

  __syncthreads();
  if (tid == 0 && *abort_flag) atomicOr(&rv.state[ST_ERR], DEVERR_TIMEOUT);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

cudaError_t prepare_attend(int D) {
  if (D == 128)
    return cudaFuncSetAttribute(fp8_ring_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnLayout<128>::ALLOC);
  return cudaFuncSetAttribute(fp8_ring_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              AttnLayout<64>::ALLOC);
}

cudaError_t launch_fp8_ring_attn(const RingView& rv, const AttnMaps& maps, const void* q, const int32_t* q_pos,
                                 int n_q, void* out, int out_f32, cudaStream_t st) {
  const dim3 grid((n_q + BM - 1) / BM, rv.H);
  if (rv.D == 128)
    fp8_ring_attn_kernel<128><<<grid, ATT_THREADS, AttnLayout<128>::ALLOC, st>>>(
        maps.k_codes, maps.v_codes, maps.k_scale, maps.v_scale, rv, static_cast<const uint4*>(q), q_pos, n_q, out,
        out_f32);
  else
    fp8_ring_attn_kernel<64><<<grid, ATT_THREADS, AttnLayout<64>::ALLOC, st>>>(
        maps.k_codes, maps.v_codes, maps.k_scale, maps.v_scale, rv, static_cast<const uint4*>(q), q_pos, n_q, out,
        out_f32);
  return cudaGetLastError();
}

}  // namespace kvring_dev
