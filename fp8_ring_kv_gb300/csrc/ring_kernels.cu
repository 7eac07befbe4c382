// ring_kv_write and delta_rerotate: the two memory-bound kernels of the ring.
//
// Runway Characters paper, §4.1 (ring cache with a device-side write
// position), §4.2 (RoPE at write; delta rotation at reset), §4.3 (FP8 at
// write), Appendix G (cache update and position reset).
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
// Block = T tokens x {K, V} x H heads x L lanes (thread order: token, kv,
// head, lane), so the threads of one (token, kv) cover that token's H*D bf16
// contiguously.  A K thread reads the cos/sin of its own 8 pairs (the token's
// table row is shared by all heads through L1); there is no block barrier.
template <int L>
__global__ void __launch_bounds__(1024) ring_kv_write_kernel(RingView rv, const uint4* __restrict__ k,
                                                             const uint4* __restrict__ v,
                                                             const int32_t* __restrict__ pos, int n_new, int T) {
  constexpr int D = L * 16;
  const int H = rv.H;
  const int t0 = blockIdx.x * T;
  const int wp = rv.state[ST_WP];

  // This thread's 32 bytes of K or V go out first: they depend on nothing
  // below, and the table gather and the barrier would otherwise delay them.
  const int per_tok = 2 * H * L;
  const int tl = threadIdx.x / per_tok;
  const int rem = threadIdx.x - tl * per_tok;
  const int kv = rem / (H * L);
  const int h = (rem / L) % H;
  const int lane = rem % L;
  const int tok = t0 + tl;
  uint4 a = make_uint4(0, 0, 0, 0), b = a;
  if (tok < n_new) {
    const uint4* src = (kv ? v : k) + ((size_t)tok * H + h) * (D / 8) + lane * 2;
    a = __ldg(src);
    b = __ldg(src + 1);
  }

  bool bad = false;
  float2 cs[8];
  if (kv == 0 && tok < n_new) {
    const int32_t* pr = pos + (size_t)tok * rv.n_axes;
#pragma unroll
    for (int m = 0; m < 8; ++m) cs[m] = rope_cs(rv, pr, lane * 8 + m, bad);
  }
  if (bad) atomicOr(&rv.state[ST_ERR], DEVERR_POS_RANGE);

  if (tok < n_new) {  // uniform over the L lanes of a row
    float x[16];
    bf16x8_to_f32(a, x);
    bf16x8_to_f32(b, x + 8);
    if (kv == 0) {
#pragma unroll
      for (int m = 0; m < 8; ++m) rope_pair(x[2 * m], x[2 * m + 1], cs[m].x, cs[m].y);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = row_max<L>(amax, row_group_mask<L>());
    float scale, inv;
    absmax_scale(amax, scale, inv);
    const uint4 codes = quant16(x, inv);
    const int slot = (int)(((long long)wp + tok) % rv.S);
    uint8_t* dst = (kv ? rv.v_codes : rv.k_codes) + ((size_t)h * rv.S + slot) * D + lane * 16;
    *reinterpret_cast<uint4*>(dst) = codes;
    if (lane == 0) (kv ? rv.v_scale : rv.k_scale)[(size_t)h * rv.S_pad + slot] = scale;
  }

  // The last block to finish advances the ring state.  Every block read wp
  // before arriving here, so the update cannot race with a reader.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int done = atomicAdd(&rv.state[ST_DONE], 1);
    if (done == (int)gridDim.x - 1) {
      rv.state[ST_WP] = (int)(((long long)wp + n_new) % rv.S);
      rv.state[ST_NVALID] = min(rv.state[ST_NVALID] + n_new, rv.S);
      rv.state[ST_DONE] = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------- query preparation
// The queries of one attention call: RoPE in fp32 at their positions and
// e4m3 with one absmax scale per (query, head), into the workspace's query
// scratch (codes [n_q][H][D], scales [H][Q_pad]) that the attention kernel
// then loads by TMA.  Same thread layout and arithmetic as the K side of
// ring_kv_write.
template <int L>
__global__ void __launch_bounds__(256) q_prep_kernel(RingView rv, const uint4* __restrict__ q,
                                                     const int32_t* __restrict__ pos, int n_q) {
  constexpr int D = L * 16;
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gt / L;            // = query * H + head
  const int lane = (int)(gt % L);
  if (row >= (long long)n_q * rv.H) return;  // whole rows
  const int qi = (int)(row / rv.H);
  const int h = (int)(row % rv.H);
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
#pragma unroll
  for (int m = 0; m < 8; ++m) rope_pair(x[2 * m], x[2 * m + 1], cs[m].x, cs[m].y);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = row_max<L>(amax, __activemask() & row_group_mask<L>());
  float scale, inv;
  absmax_scale(amax, scale, inv);
  *reinterpret_cast<uint4*>(rv.q_codes + row * D + lane * 16) = quant16(x, inv);
  if (lane == 0) rv.q_scale[(size_t)h * rv.Q_pad + qi] = scale;
}

// ---------------------------------------------------------------- delta_rerotate
// One thread per 16 codes of a key row, over rows (head, slot) with
// slot < n_valid.  In place: dequantise (code * scale, fp32), rotate the
// temporal pairs by the host-computed (cos, sin) of -d * omega_j, re-quantise
// with a fresh absmax scale.
template <int L>
__global__ void __launch_bounds__(256) delta_rerotate_kernel(RingView rv, DeltaTable dt) {
  constexpr int D = L * 16;
  // the lanes of a warp read 8 different pairs at once: from shared memory,
  // not from the parameter space (which would serialise them)
  __shared__ float2 cs_s[64];
  if (threadIdx.x < 64) cs_s[threadIdx.x] = dt.cs[threadIdx.x];
  __syncthreads();
  const int n_valid = rv.state[ST_NVALID];
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gt / L;
  const int lane = (int)(gt % L);
  if (row >= (long long)rv.H * rv.S) return;  // whole rows
  const int h = (int)(row / rv.S);
  const int slot = (int)(row % rv.S);
  if (slot >= n_valid) return;                // whole rows
  uint8_t* p = rv.k_codes + ((size_t)h * rv.S + slot) * D + lane * 16;
  float* sp = rv.k_scale + (size_t)h * rv.S_pad + slot;
  const uint4 c = *reinterpret_cast<const uint4*>(p);
  const float scale = *sp;
  float x[16];
  dequant16_codes(c, x);
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = __fmul_rn(x[i], scale);
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int pr = lane * 8 + m;
    if (pr < dt.n_pairs) {
      const float2 c = cs_s[pr];
      rope_pair(x[2 * m], x[2 * m + 1], c.x, c.y);
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const unsigned mask = __activemask();
  amax = row_max<L>(amax, mask & row_group_mask<L>());
  float nscale, inv;
  absmax_scale(amax, nscale, inv);
  *reinterpret_cast<uint4*>(p) = quant16(x, inv);
  if (lane == 0) *sp = nscale;
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
  amax = row_max<L>(amax, __activemask() & row_group_mask<L>());
  float scale, inv;
  absmax_scale(amax, scale, inv);
  *reinterpret_cast<uint4*>(codes + row * D + lane * 16) = quant16(v, inv);
  if (lane == 0) scales[row] = scale;
}

// ---------------------------------------------------------------- launchers
template <int L>
static cudaError_t launch_write_t(const RingView& rv, const void* k, const void* v, const int32_t* pos, int n_new,
                                  cudaStream_t st) {
  const int per_tok = 2 * rv.H * L;
  int T = 256 / per_tok;
  if (T < 1) T = 1;
  const int threads = per_tok * T;
  const int blocks = (n_new + T - 1) / T;
  ring_kv_write_kernel<L><<<blocks, threads, 0, st>>>(rv, static_cast<const uint4*>(k),
                                                         static_cast<const uint4*>(v), pos, n_new, T);
  return cudaGetLastError();
}

cudaError_t launch_ring_kv_write(const RingView& rv, const void* k, const void* v, const int32_t* pos, int n_new,
                                 cudaStream_t st) {
  if (rv.D == 64) return launch_write_t<4>(rv, k, v, pos, n_new, st);
  return launch_write_t<8>(rv, k, v, pos, n_new, st);
}

cudaError_t launch_q_prep(const RingView& rv, const void* q, const int32_t* q_pos, int n_q, cudaStream_t st) {
  const int L = rv.D / 16;
  const long long threads = (long long)n_q * rv.H * L;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (L == 4)
    q_prep_kernel<4><<<blocks, 256, 0, st>>>(rv, static_cast<const uint4*>(q), q_pos, n_q);
  else
    q_prep_kernel<8><<<blocks, 256, 0, st>>>(rv, static_cast<const uint4*>(q), q_pos, n_q);
  return cudaGetLastError();
}

cudaError_t launch_delta_rerotate(const RingView& rv, const DeltaTable& dt, cudaStream_t st) {
  const int L = rv.D / 16;
  const long long threads = (long long)rv.H * rv.S * L;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (L == 4)
    delta_rerotate_kernel<4><<<blocks, 256, 0, st>>>(rv, dt);
  else
    delta_rerotate_kernel<8><<<blocks, 256, 0, st>>>(rv, dt);
  return cudaGetLastError();
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
