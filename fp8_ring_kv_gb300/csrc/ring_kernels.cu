// ring_kv_write and delta_rerotate: the two memory-bound kernels of the ring.
//
// Runway Characters paper, §4.1 (ring cache with a device-side write
// position), §4.2 (RoPE at write; delta rotation at reset), §4.3 (FP8 at
// write), Appendix G (cache update and position reset).
//
// Slots 0 .. G-1 hold the session's global tokens (written once, never
// rotated); the window ring is slots G .. S-1, W = S - G of them (G = 0: the
// whole cache is the ring).
//
// Both kernels stream rows of one (token or slot, head): a row of D channels
// is handled by L = D/16 consecutive lanes, each owning 16 channels (32 bytes
// of bf16 in, 16 bytes of e4m3 out), so every global access is a full 16-byte
// vector and a warp covers whole 128-byte lines.  The row's absolute maximum
// is reduced with L-lane shuffles.
#include "common.cuh"
#include "launch.h"

namespace kvring_dev {

template <int L>
__device__ __forceinline__ float row_max(float v, unsigned group_mask) {
#pragma unroll
  for (int off = L / 2; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(group_mask, v, off));
  return v;
}

template <int L>
__device__ __forceinline__ unsigned row_group_mask() {
  const unsigned lane = threadIdx.x & 31u;
  const unsigned base = lane & ~(unsigned)(L - 1);
  return (L == 32 ? 0xFFFFFFFFu : ((1u << L) - 1u)) << base;
}

// ---------------------------------------------------------------- ring_kv_write
// Block = T tokens x H heads x L lanes (thread order: token, head, lane); a
// thread owns 16 channels of one (token, head) and writes both its K and its
// V codes, so the threads of one token cover that token's H*D bf16 of K and
// of V contiguously.  The inputs, positions and cos/sin are loaded before
// anything is read from the ring.  Thread 0 reads the write position once for
// the block; as soon as it has, the block counts itself in, and the last
// block to do so advances the ring state (every block has read the position
// by then).  No barrier waits for the stores.
//
// Window write: token i goes to slot G + (wp + i) mod W; then wp <- (wp + N)
// mod W and n_valid <- min(n_valid + N, S).  Global write (``glob``, the G
// global tokens, once): token i goes to slot i; then n_valid <- N.
//
// Scales: per (token, head) absmax; on a ring with per-head fixed scales
// (scale_mode 1) the same until calibration, with each row's maximum also
// folded into its head's recorded maximum, and after it the head's fixed
// (scale, inv), values beyond the range saturating.
template <int L, bool kNorm>
__global__ void __launch_bounds__(512, 2) ring_kv_write_kernel(RingView rv, const uint4* __restrict__ k,
                                                               const uint4* __restrict__ v,
                                                               const int32_t* __restrict__ pos, int n_new, int T,
                                                               bool glob) {
  constexpr int D = L * 16;
  __shared__ int wp_s;
  const int H = rv.H;
  const int per_tok = H * L;
  const int tl = threadIdx.x / per_tok;
  const int rem = threadIdx.x - tl * per_tok;
  const int h = rem / L;
  const int lane = rem % L;
  const int tok = blockIdx.x * T + tl;
  const bool live = tok < n_new;   // uniform over the L lanes of a row
  pdl_wait();
  pdl_trigger();
  // the write position (and mode) first, so that its latency overlaps the
  // input loads below
  int wp0 = 0, fixed0 = 0;
  if (threadIdx.x == 0) {
    wp0 = rv.state[ST_WP];
    fixed0 = rv.scale_mode ? rv.state[ST_STATIC] : 0;
  }

  uint4 ka = make_uint4(0, 0, 0, 0), kb = ka, va = ka, vb = ka;
  if (live) {
    const size_t off = ((size_t)tok * H + h) * (D / 8) + lane * 2;
    ka = __ldg(k + off);
    kb = __ldg(k + off + 1);
    va = __ldg(v + off);
    vb = __ldg(v + off + 1);
  }
  bool bad = false;
  float2 cs[8];
  if (live) {
    const int32_t* pr = pos + (size_t)tok * rv.n_axes;
#pragma unroll
    for (int m = 0; m < 8; ++m) cs[m] = rope_cs(rv, pr, lane * 8 + m, bad);
  }
  if (bad) atomicOr(&rv.state[ST_ERR], DEVERR_POS_RANGE);

  __shared__ int fixed_s;
  if (threadIdx.x == 0) {
    wp_s = wp0;
    fixed_s = fixed0;
  }
  __syncthreads();
  const int wp = wp_s;
  const bool fixed = fixed_s != 0;
  const int W = rv.S - rv.G;
  if (threadIdx.x == 0) {
    const int done = atomicAdd(&rv.state[ST_DONE], 1);
    if (done == (int)gridDim.x - 1) {
      if (glob) {
        rv.state[ST_NVALID] = n_new;
      } else {
        rv.state[ST_WP] = (int)(((long long)wp + n_new) % W);
        rv.state[ST_NVALID] = min(rv.state[ST_NVALID] + n_new, rv.S);
      }
      rv.state[ST_DONE] = 0;
    }
  }
  if (!live) return;

  const int slot = glob ? tok : rv.G + (int)(((long long)wp + tok) % W);
  const size_t row = (size_t)h * rv.S + slot;
  const unsigned gm = row_group_mask<L>();
  {
    float x[16];
    bf16x8_to_f32(ka, x);
    bf16x8_to_f32(kb, x + 8);
    if constexpr (kNorm) rms_norm16<L>(x, rv.gamma_k + (size_t)h * (D / 8) + lane * 2, rv.norm_eps, gm);
#pragma unroll
    for (int m = 0; m < 8; ++m) rope_pair(x[2 * m], x[2 * m + 1], cs[m].x, cs[m].y);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = row_max<L>(amax, gm);
    float scale, inv;
    row_absmax_scale<L>(amax, scale, inv, gm);
    if (fixed) {
      scale = rv.stat[STAT_K_SCALE * rv.H + h];
      inv = rv.stat[STAT_K_INV * rv.H + h];
    } else if (rv.scale_mode && lane == 0) {
      atomicMax(reinterpret_cast<int*>(rv.stat) + STAT_AMAX_K * rv.H + h, __float_as_int(amax));
    }
    *reinterpret_cast<uint4*>(rv.k_codes + row * D + lane * 16) = quant16(x, inv);
    if (lane == 0) rv.k_scale[(size_t)h * rv.S_pad + slot] = scale;
  }
  {
    float x[16];
    bf16x8_to_f32(va, x);
    bf16x8_to_f32(vb, x + 8);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = row_max<L>(amax, gm);
    float scale, inv;
    row_absmax_scale<L>(amax, scale, inv, gm);
    if (fixed) {
      scale = rv.stat[STAT_V_SCALE * rv.H + h];
      inv = rv.stat[STAT_V_INV * rv.H + h];
    } else if (rv.scale_mode && lane == 0) {
      atomicMax(reinterpret_cast<int*>(rv.stat) + STAT_AMAX_V * rv.H + h, __float_as_int(amax));
    }
    *reinterpret_cast<uint4*>(rv.v_codes + row * D + lane * 16) = quant16(x, inv);
    if (lane == 0) rv.v_scale[(size_t)h * rv.S_pad + slot] = scale;
  }
}

// ---------------------------------------------------------------- query preparation
// The queries of one attention call: RoPE in fp32 at their positions and
// e4m3 with one absmax scale per (query, head), into the workspace's query
// scratch (codes [n_q][H][D], scales [H][Q_pad]) that the attention kernel
// then loads by TMA.  Same thread layout (T queries x H heads x L lanes per
// block) and arithmetic as the K side of ring_kv_write (with the RMS norm of
// Q first when the ring has Q norm weights).
//
// Blocks past the queries' (one per head, blockIdx.x = n_qblocks + h) find
// the head's largest V scale over the valid slots and store the attention's
// per-head range factor and scale floor (attn_head_factors) in the scratch.
template <int L, bool kNorm>
__global__ void __launch_bounds__(512, 2) q_prep_kernel(RingView rv, const uint4* __restrict__ q,
                                                        const int32_t* __restrict__ pos, int n_q, int T,
                                                        int n_qblocks) {
  constexpr int D = L * 16;
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x >= n_qblocks) {
    __shared__ float wmax[16];
    const int h = blockIdx.x - n_qblocks;
    const int n_valid = rv.state[ST_NVALID];
    // each head's scale row starts 16-byte aligned (rows are S_pad, a
    // multiple of 4, apart)
    const float* vs1 = rv.v_scale + (size_t)h * rv.S_pad;
    const float4* vs = reinterpret_cast<const float4*>(vs1);
    const int n4 = n_valid >> 2;
    float mx = 0.0f;
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      const float4 v = __ldg(vs + i);
      mx = fmaxf(mx, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
    }
    if ((int)threadIdx.x < (n_valid & 3)) mx = fmaxf(mx, vs1[n4 * 4 + threadIdx.x]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    const int nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < nw; ++w) mx = fmaxf(mx, wmax[w]);
      float c, fl;
      attn_head_factors(mx, c, fl);
      rv.head_stat[2 * h] = c;
      rv.head_stat[2 * h + 1] = fl;
    }
    return;
  }
  const int per_q = rv.H * L;
  const int tl = threadIdx.x / per_q;
  const int rem = threadIdx.x - tl * per_q;
  const int h = rem / L;
  const int lane = rem % L;
  const int qi = blockIdx.x * T + tl;
  if (qi >= n_q) return;   // whole rows
  const size_t row = (size_t)qi * rv.H + h;
  const uint4* src = q + row * (D / 8) + lane * 2;
  const uint4 a = __ldg(src);
  const uint4 b = __ldg(src + 1);
  bool bad = false;
  float2 cs[8];
  const int32_t* pr = pos + (size_t)qi * rv.n_axes;
#pragma unroll
  for (int m = 0; m < 8; ++m) cs[m] = rope_cs(rv, pr, lane * 8 + m, bad);
  if (bad) atomicOr(&rv.state[ST_ERR], DEVERR_POS_RANGE);
  float x[16];
  bf16x8_to_f32(a, x);
  bf16x8_to_f32(b, x + 8);
  if constexpr (kNorm) rms_norm16<L>(x, rv.gamma_q + (size_t)h * (D / 8) + lane * 2, rv.norm_eps, row_group_mask<L>());
#pragma unroll
  for (int m = 0; m < 8; ++m) rope_pair(x[2 * m], x[2 * m + 1], cs[m].x, cs[m].y);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = row_max<L>(amax, row_group_mask<L>());
  float scale, inv;
  row_absmax_scale<L>(amax, scale, inv, row_group_mask<L>());
  *reinterpret_cast<uint4*>(rv.q_codes + row * D + lane * 16) = quant16(x, inv);
  if (lane == 0) rv.q_scale[(size_t)h * rv.Q_pad + qi] = scale;
}

// ---------------------------------------------------------------- delta_rerotate
// In place over the window's key rows (head, slot), G <= slot < n_valid
// (the global keys keep their positions), on a calibrated ring with per-head
// fixed scales re-quantised with the head's scale (saturating: the clamp)
// instead of a fresh one: dequantise
// (code * scale, fp32), rotate the temporal pairs by the host-computed
// (cos, sin) of -d * omega_j, re-quantise with a fresh absmax scale.  A row
// is L lanes of 16 codes; the grid is sized to stay resident and each thread
// walks rows with a stride of the whole grid, loading its next 16 codes and
// scale before working on the current ones so that two loads are in flight.
//
// The walk over one ring, for thread ``first`` of ``stride`` threads that
// share the ring (cs_s: the rotation's (cos, sin) per temporal pair, in
// shared memory: the lanes of a warp read 8 different pairs at once).
template <int L>
__device__ __forceinline__ void rerotate_ring(const RotRing& rv, const float2* cs_s, int n_pairs, int first,
                                              int stride) {
  constexpr int D = L * 16;
  // rows are walked as (h, s) over the n_win valid window slots, s = slot - G
  const int n_win = rv.state[ST_NVALID] - rv.G;
  if (n_win <= 0) return;
  const bool fixed = rv.scale_mode && rv.state[ST_STATIC];
  const int chunks = rv.H * n_win * L;            // <= 128 heads x 2^20 slots x 8
  const int lane = threadIdx.x % L;               // stride and first are multiples of 32: rows never split
  // pairs past the temporal axis are left as they are (not rotated by the
  // identity, which would turn a -0 into +0)
  float2 cs[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) cs[m] = cs_s[(lane * 8 + m) & 63];
  // the thread's row (head h, slot) advances by a fixed number of rows per
  // step: kept as (h, slot) and carried, instead of two divisions per row
  const int row_step = stride / L;
  const int step_h = row_step / n_win;
  const int step_slot = row_step - step_h * n_win;
  int c = first;
  if (c >= chunks) return;   // whole rows
  int h = (c / L) / n_win;
  int slot = c / L - h * n_win;
  auto locate = [&](int hh, int ss, uint8_t*& p, float*& sp) {
    p = rv.k_codes + ((size_t)hh * rv.S + rv.G + ss) * D + lane * 16;
    sp = rv.k_scale + (size_t)hh * rv.S_pad + rv.G + ss;
  };
  uint8_t* p;
  float* sp;
  locate(h, slot, p, sp);
  uint4 code = *reinterpret_cast<const uint4*>(p);
  float scale = *sp;
  while (true) {
    const int cn = c + stride;
    const bool more = cn < chunks;   // whole rows
    uint8_t* pn = p;
    float* spn = sp;
    uint4 code_n = code;
    float scale_n = scale;
    int hn = h + step_h, sn = slot + step_slot;
    if (sn >= n_win) {
      sn -= n_win;
      ++hn;
    }
    if (more) {
      locate(hn, sn, pn, spn);
      code_n = *reinterpret_cast<const uint4*>(pn);
      scale_n = *spn;
    }
    float x[16];
    dequant16_scaled(code, scale, x);
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if (lane * 8 + m < n_pairs) rope_pair(x[2 * m], x[2 * m + 1], cs[m].x, cs[m].y);
    if (fixed) {
      // the head's scale is kept; values beyond its range saturate
      *reinterpret_cast<uint4*>(p) = quant16(x, rv.stat[STAT_K_INV * rv.H + h]);
    } else {
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
      amax = row_max<L>(amax, row_group_mask<L>());
      float nscale, inv;
      row_absmax_scale<L>(amax, nscale, inv, row_group_mask<L>());
      *reinterpret_cast<uint4*>(p) = quant16(x, inv);
      if (lane == 0) *sp = nscale;
    }
    if (!more) break;
    c = cn;
    h = hn;
    slot = sn;
    p = pn;
    sp = spn;
    code = code_n;
    scale = scale_n;
  }
}

template <int L>
__global__ void __launch_bounds__(256, 4) delta_rerotate_kernel(RotRing rr, DeltaTable dt) {
  __shared__ float2 cs_s[64];
  if (threadIdx.x < 64) cs_s[threadIdx.x] = dt.cs[threadIdx.x];
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  rerotate_ring<L>(rr, cs_s, dt.n_pairs, blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x);
}

// Several rings in one launch (the rings of every layer at a position reset):
// blockIdx.y is the ring, the blocks along x share its rows.
template <int L>
__global__ void __launch_bounds__(256, 4) delta_rerotate_batch_kernel(const __grid_constant__ RotBatch rb,
                                                                      DeltaTable dt) {
  __shared__ float2 cs_s[64];
  if (threadIdx.x < 64) cs_s[threadIdx.x] = dt.cs[threadIdx.x];
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  rerotate_ring<L>(rb.r[blockIdx.y], cs_s, dt.n_pairs, blockIdx.x * blockDim.x + threadIdx.x,
                   gridDim.x * blockDim.x);
}

// ---------------------------------------------------------------- calibration
// Per-head fixed scales from the recorded maxima (paper §4.3, Appendix G):
// a = fl32(margin * amax), scale = fl32(a / 448), inv = fl32(448 / a), both
// 0 when a = 0.  One thread per (tensor, head); marks the ring calibrated.
__global__ void calib_scales_kernel(RingView rv, float margin) {
  const int t = threadIdx.x;   // 0 .. 2H-1: K heads, then V heads
  if (t < 2 * rv.H) {
    const int v = t >= rv.H;
    const int h = t - v * rv.H;
    const float amax = rv.stat[(v ? STAT_AMAX_V : STAT_AMAX_K) * rv.H + h];
    const float a = __fmul_rn(margin, amax);
    const float scale = a > 0.0f ? __fdiv_rn(a, kE4m3Max) : 0.0f;
    const float inv = a > 0.0f ? __fdiv_rn(kE4m3Max, a) : 0.0f;
    rv.stat[(v ? STAT_V_SCALE : STAT_K_SCALE) * rv.H + h] = scale;
    rv.stat[(v ? STAT_V_INV : STAT_K_INV) * rv.H + h] = inv;
  }
  if (t == 0) rv.state[ST_STATIC] = 1;
}

// Every valid K and V row, re-quantised with its head's fixed scale from its
// dequantised value (code * scale, fp32); the row's scale entry becomes the
// head's.  A row is L lanes of 16 codes; grid-stride over (tensor, head, slot).
template <int L>
__global__ void __launch_bounds__(256) calib_requant_kernel(RingView rv) {
  constexpr int D = L * 16;
  const int n_valid = rv.state[ST_NVALID];
  const long long rows = 2LL * rv.H * n_valid;
  const int lane = threadIdx.x % L;
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / L; r < rows;
       r += (long long)gridDim.x * blockDim.x / L) {
    const int v = (int)(r / ((long long)rv.H * n_valid));
    const int rem = (int)(r - (long long)v * rv.H * n_valid);
    const int h = rem / n_valid;
    const int slot = rem - h * n_valid;
    uint8_t* p = (v ? rv.v_codes : rv.k_codes) + ((size_t)h * rv.S + slot) * D + lane * 16;
    float* sp = (v ? rv.v_scale : rv.k_scale) + (size_t)h * rv.S_pad + slot;
    const float old = *sp;
    float x[16];
    dequant16_scaled(*reinterpret_cast<const uint4*>(p), old, x);
    *reinterpret_cast<uint4*>(p) = quant16(x, rv.stat[(v ? STAT_V_INV : STAT_K_INV) * rv.H + h]);
    __syncwarp(row_group_mask<L>());   // every lane has read the old scale before lane 0 replaces it
    if (lane == 0) *sp = rv.stat[(v ? STAT_V_SCALE : STAT_K_SCALE) * rv.H + h];
  }
}

cudaError_t launch_calibrate(const RingView& rv, float margin, cudaStream_t st) {
  calib_scales_kernel<<<1, 256, 0, st>>>(rv, margin);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int L = rv.D / 16;
  // enough threads for one pass over a full ring's K and V rows, at most 8
  // blocks of 256 per SM (the kernel strides over the rest)
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  long long blocks = (2LL * rv.H * rv.S * L + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  if (blocks < 1) blocks = 1;
  if (L == 4)
    calib_requant_kernel<4><<<(unsigned)blocks, 256, 0, st>>>(rv);
  else
    calib_requant_kernel<8><<<(unsigned)blocks, 256, 0, st>>>(rv);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- bounded wait
// The kernels' barrier wait as it is used everywhere (warp_wait: every lane
// waits, one answer per warp), on a barrier of two arrivals that gets one --
// or, with ``complete``, both.  A wait that gives up raises the block's abort
// flag; the block then records DEVERR_TIMEOUT and how long it waited, and
// returns.  Nothing else is left pending: no copy or MMA was issued.
__global__ void __launch_bounds__(64) debug_wait_kernel(long long limit_ns, int complete, int64_t* out2) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 2);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(&bar);
    if (complete) mbar_arrive(&bar);
  }
  const unsigned long long t0 = globaltimer_ns();
  const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar, 0, &abort_flag, (unsigned long long)limit_ns));
  const unsigned long long t1 = globaltimer_ns();
  __syncthreads();
  if (threadIdx.x == 0) {
    out2[0] = (ok && !abort_flag) ? 0 : DEVERR_TIMEOUT;
    out2[1] = (int64_t)(t1 - t0);
  }
}

cudaError_t launch_debug_wait(long long limit_ns, bool complete, int64_t* out2, cudaStream_t st) {
  debug_wait_kernel<<<1, 64, 0, st>>>(limit_ns, complete ? 1 : 0, out2);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- debug quantiser
template <int L>
__global__ void __launch_bounds__(256) debug_quantize_kernel(const float* __restrict__ x, long long rows,
                                                             uint8_t* __restrict__ codes, float* __restrict__ scales) {
  constexpr int D = L * 16;
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gt / L;
  const int lane = (int)(gt % L);
  if (row >= rows) return;  // whole rows
  const float4* src = reinterpret_cast<const float4*>(x + row * D + lane * 16);
  float v[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = src[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = row_max<L>(amax, row_group_mask<L>());
  float scale, inv;
  row_absmax_scale<L>(amax, scale, inv, row_group_mask<L>());
  *reinterpret_cast<uint4*>(codes + row * D + lane * 16) = quant16(v, inv);
  if (lane == 0) scales[row] = scale;
}

// ---------------------------------------------------------------- launchers
template <int L>
static cudaError_t launch_write_t(const RingView& rv, const void* k, const void* v, const int32_t* pos, int n_new,
                                  bool glob, cudaStream_t st) {
  const int per_tok = rv.H * L;
  int T = 192 / per_tok;
  if (T < 1) T = 1;
  const int threads = per_tok * T;
  const int blocks = (n_new + T - 1) / T;
  if (rv.gamma_k)
    return launch_pdl(ring_kv_write_kernel<L, true>, dim3(blocks), dim3(threads), 0, st, rv,
                      static_cast<const uint4*>(k), static_cast<const uint4*>(v), pos, n_new, T, glob);
  return launch_pdl(ring_kv_write_kernel<L, false>, dim3(blocks), dim3(threads), 0, st, rv,
                    static_cast<const uint4*>(k), static_cast<const uint4*>(v), pos, n_new, T, glob);
}

cudaError_t launch_ring_kv_write(const RingView& rv, const void* k, const void* v, const int32_t* pos, int n_new,
                                 bool glob, cudaStream_t st) {
  if (rv.D == 64) return launch_write_t<4>(rv, k, v, pos, n_new, glob, st);
  return launch_write_t<8>(rv, k, v, pos, n_new, glob, st);
}

cudaError_t launch_q_prep(const RingView& rv, const void* q, const int32_t* q_pos, int n_q, cudaStream_t st) {
  const int L = rv.D / 16;
  const int per_q = rv.H * L;
  int T = 192 / per_q;
  if (T < 1) T = 1;
  const int qblocks = (n_q + T - 1) / T;
  const dim3 grid(qblocks + rv.H), block(per_q * T);   // then one block per head: the range factors
  const uint4* qq = static_cast<const uint4*>(q);
  if (L == 4)
    return rv.gamma_q ? launch_pdl(q_prep_kernel<4, true>, grid, block, 0, st, rv, qq, q_pos, n_q, T, qblocks)
                      : launch_pdl(q_prep_kernel<4, false>, grid, block, 0, st, rv, qq, q_pos, n_q, T, qblocks);
  return rv.gamma_q ? launch_pdl(q_prep_kernel<8, true>, grid, block, 0, st, rv, qq, q_pos, n_q, T, qblocks)
                    : launch_pdl(q_prep_kernel<8, false>, grid, block, 0, st, rv, qq, q_pos, n_q, T, qblocks);
}

// Blocks that stay resident on every SM at once (computed once per process).
template <int L>
static int rerotate_grid() {
  static int blocks = 0;
  if (blocks == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, delta_rerotate_kernel<L>, 256, 0) != cudaSuccess ||
        sms <= 0 || per_sm <= 0)
      return 0;
    blocks = sms * per_sm;
  }
  return blocks;
}

RotRing rot_ring(const RingView& rv) {
  RotRing r{};
  r.k_codes = rv.k_codes;
  r.k_scale = rv.k_scale;
  r.state = rv.state;
  r.stat = rv.stat;
  r.H = rv.H;
  r.S = rv.S;
  r.S_pad = rv.S_pad;
  r.G = rv.G;
  r.scale_mode = rv.scale_mode;
  return r;
}

cudaError_t launch_delta_rerotate(const RingView& rv, const DeltaTable& dt, cudaStream_t st) {
  const int L = rv.D / 16;
  // enough threads for one pass over a full ring, at most what stays resident
  const long long need = ((long long)rv.H * rv.S * L + 255) / 256;
  const int resident = L == 4 ? rerotate_grid<4>() : rerotate_grid<8>();
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const unsigned blocks = (unsigned)(need < resident ? need : resident);
  const RotRing rr = rot_ring(rv);
  if (L == 4) return launch_pdl(delta_rerotate_kernel<4>, dim3(blocks), dim3(256), 0, st, rr, dt);
  return launch_pdl(delta_rerotate_kernel<8>, dim3(blocks), dim3(256), 0, st, rr, dt);
}

cudaError_t launch_delta_rerotate_batch(const RingView* const* rvs, int n, const DeltaTable& dt, cudaStream_t st) {
  if (n < 1) return cudaSuccess;
  const int L = rvs[0]->D / 16;
  const int resident = L == 4 ? rerotate_grid<4>() : rerotate_grid<8>();
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  for (int i0 = 0; i0 < n; i0 += kMaxBatchRings) {
    const int m = n - i0 < kMaxBatchRings ? n - i0 : kMaxBatchRings;
    RotBatch rb{};
    long long need = 1;
    for (int i = 0; i < m; ++i) {
      rb.r[i] = rot_ring(*rvs[i0 + i]);
      const long long ni = ((long long)rvs[i0 + i]->H * rvs[i0 + i]->S * L + 255) / 256;
      need = ni > need ? ni : need;
    }
    // the resident grid shared among the rings of the launch
    long long per = resident / m;
    if (per < 1) per = 1;
    const unsigned bx = (unsigned)(need < per ? need : per);
    const cudaError_t e =
        L == 4 ? launch_pdl(delta_rerotate_batch_kernel<4>, dim3(bx, m), dim3(256), 0, st, rb, dt)
               : launch_pdl(delta_rerotate_batch_kernel<8>, dim3(bx, m), dim3(256), 0, st, rb, dt);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_debug_quantize(const float* x, long long rows, int d, uint8_t* codes, float* scales,
                                  cudaStream_t st) {
  const int L = d / 16;
  const long long threads = rows * L;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  switch (L) {
    case 1: debug_quantize_kernel<1><<<blocks, 256, 0, st>>>(x, rows, codes, scales); break;
    case 2: debug_quantize_kernel<2><<<blocks, 256, 0, st>>>(x, rows, codes, scales); break;
    case 4: debug_quantize_kernel<4><<<blocks, 256, 0, st>>>(x, rows, codes, scales); break;
    case 8: debug_quantize_kernel<8><<<blocks, 256, 0, st>>>(x, rows, codes, scales); break;
    case 16: debug_quantize_kernel<16><<<blocks, 256, 0, st>>>(x, rows, codes, scales); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kvring_dev
