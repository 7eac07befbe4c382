// fp8_ring_attn: n_q queries attend over every valid slot of the FP8 ring.
//
// Runway Characters paper, §4.3 (K and V stored as float8_e4m3, the queries
// quantised per call, attention reading the FP8 cache directly) and
// Appendix G (each call reads all the cache's slots; no causal mask).
//
// The queries arrive rotated and e4m3-coded, with one scale per (query,
// head), from the query preparation kernel, which also leaves two per-head
// numbers (the range factor c and the scale floor, below) next to them.  One
// block per (tile of 128 queries, head).  The slots are visited in tiles of
// 128 in storage order: attention is a sum over the valid slots, so the ring's
// wrap needs no reordering, and slots >= n_valid are masked.
//
//   S_j  = Qcodes . Kcodes_j^T            tcgen05 kind::f8f6f4, fp32 in TMEM
//   t    = S_j * s_k (per column);  logit*log2(e) = t * s_q * log2(e)/sqrt(D)
//   online softmax in base 2: e = exp2(t*r - m + c), with a running row
//   maximum m that is only raised (and O, L rescaled) when a tile's maximum
//   exceeds it by more than 2^kLazyLog2
//   P_j  = e * w (per column, w = max(s_v, floor)) rounded to fp16, in TMEM
//   [O | L] += P_j . [Vcodes_j | u_hi | u_lo | 0]   tcgen05 kind::f16, N = D + 16
//                                          (A = P from TMEM; u = 2^-c / w)
//   out  = O / (L * 2^c)
// The e4m3 V codes are widened to fp16 in shared memory (exact) because the
// fp16 MMA takes both operands in fp16; P in fp16 keeps the weighted sum of V
// within the accuracy that e4m3 weights would lose.  2^c is a per-head power of
// two (cancelling between O and L) that keeps P within fp16 range.
//
// The row sums are taken from the same fp16 P as the weighted sum of V (u
// split into two fp16 parts, u_hi + u_lo * 2^-11, good to about 2^-22), so the
// rounding of each P cancels between O and L: a row dominated by one slot
// returns that slot's value, not the value times the fp16 rounding of its
// weight (up to 2^-11 of |v|).  The per-head floor, 2^-15 * max(max s_v,
// 2^-c), keeps a zero or near-zero V row's weight in L; it changes that row's
// own (near-zero) values by at most 448 * floor.
//
// Pipeline.  TMEM holds two 128-column S buffers and the O accumulator with
// the row sums L in 16 columns after it.  The softmax of tile j loads S_j
// from buffer j % 2 into registers and stores P_j (fp16 pairs) over the first
// 64 columns of the same buffer; the MMA sequence is QK_0, QK_1, then per
// tile j: PV_j (once P_j and the fp16 V_j are in) and, once PV_j is done
// reading P_j, QK_{j+2} into that buffer.  So the softmax of tile j + 1 runs
// while PV_j and QK_{j+2} execute, and it never waits for a PV unless the
// tile raises a row maximum (O and L are then rescaled once PV_j is done).
// No MMA writes TMEM that another MMA may still read.  A tile whose maximum passes
// the bound is found before its exponentials (the row maxima are voted on
// first), so no weight can overflow.  TMEM lane quarter q can only be read by
// the warps of SM sub-partition q, so the softmax of rows 32q .. 32q+31 runs on
// that sub-partition, two warps per quarter (one per 16-lane half).
//
// Warp roles (448 threads):
//   warps 0-7   softmax: warp w serves the 16-lane half w/4 of TMEM lane
//               quarter w%4 in the 16x256b shape; finally the output, half of
//               the quarter's columns each
//   warps 8-11  per tile: the scales in the softmax's order, and the fp16
//               B operand of PV: V widened, then the u columns (one warp per
//               sub-partition)
//   warp 12     TMA producer (the e4m3 query tile, then K, V codes into
//               NSTAGE stages and, running ahead of them, their scales into
//               NSC stages)
//   warp 13     TMEM allocation and MMA issue
// Every wait is bounded (an error bit and an orderly exit after the limit);
// the TMA lane, whose loads run ahead of need, sleeps briefly whenever no
// stage can move, so that its polling leaves issue slots to the softmax.
#include <cfloat>

#include "common.cuh"
#include "launch.h"

namespace kvring_dev {

constexpr int BM = 128;           // query rows per block
constexpr int BN = kAttnKeyTile;  // slots per tile
constexpr int NSTAGE = 3;         // fp8 K/V stages
constexpr int NSC = 6;            // scale stages (held until the tile's softmax ends)
constexpr int ATT_THREADS = 448;
constexpr int SOFT_WARPS = 8;
constexpr int SOFT_THREADS = 32 * SOFT_WARPS;
constexpr int CONV_WARPS = 4;
constexpr int CONV_THREADS = 32 * CONV_WARPS;
constexpr int WARP_TMA = SOFT_WARPS + CONV_WARPS;
constexpr int WARP_MMA = WARP_TMA + 1;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;      // buffer b at columns 128 b: S fp32 [128 lanes][128], then P over it: fp16 pairs [128][64]
constexpr uint32_t TM_O = 256;    // O: fp32 [128 lanes][D], then L: columns D (hi) and D + 1 (lo) of 16
constexpr int UN = 16;            // columns of PV's N given to the row sums
// The softmax thread (c4 = lane % 4) of the 16x256b shape reads columns
// 8k + 2 c4 + e (k < 16, e < 2) of a tile; their scales are stored at
// c4 * kPermStride + 2k + e so that each thread loads 32 consecutive floats
// (8 x 16 bytes), the four groups on distinct banks.
constexpr int kPermStride = 36;
// log2 of the largest unnormalised weight.  A wider bound makes rescales (O
// and L rescaled) rarer, but the per-head factor 2^c that keeps every
// P = weight * w * 2^c below fp16's maximum then puts the row's largest P
// lower, and more of its small weights into fp16 subnormals or zero.  Those
// weights are lost to L as well as to O, and with many of them that changes
// the output.  Right after a row's maximum is set, its largest P is
// 2^(14 - kLazyLog2 - kHeadroom) = 2^0 (times w 2^c in [1, 2)), so weights
// down to 2^-14 of it stay normal.
constexpr int kLazyLog2 = kAttnLazyLog2;
constexpr float kLazyRescale = (float)kLazyLog2;
// A running maximum is set this many octaves above the tile maximum that sets
// it (weights then start at most 2^-4), so later tiles may exceed the observed
// maximum by kLazyLog2 + 4 octaves before a rescale.
constexpr float kHeadroom = 4.0f;

template <int D>
struct AttnLayout {
  static constexpr int SC_BYTES = 2 * BN * 4 + 2 * 4 * kPermStride * 4;   // raw s_k, s_v; permuted s_k, w
  static constexpr int Q = 0;                            // e4m3 [BM][D], K-major swizzled
  static constexpr int K0 = Q + BM * D;                  // NSTAGE x e4m3 [BN][D]
  static constexpr int V0 = K0 + NSTAGE * BN * D;        // NSTAGE x e4m3 [BN][D]
  // fp16 B operand of PV, MN-major, 128-byte swizzle: 64-column blocks of
  // [BN][128 bytes]; D / 64 blocks of V, then one whose columns 0, 1 hold
  // u_hi, u_lo (columns 2 .. 15 zero, the rest unused)
  static constexpr int VH_BLOCKS = D / 64 + 1;
  static constexpr int VH_BYTES = VH_BLOCKS * BN * 128;
  static constexpr int VH0 = V0 + NSTAGE * BN * D;       // 2 x VH_BYTES
  static constexpr int SC0 = VH0 + 2 * VH_BYTES;         // NSC x {s_k [BN], s_v [BN], perm s_k, perm w}
  static constexpr int BAR = SC0 + NSC * SC_BYTES;
  static constexpr int NBAR = 2 * NSTAGE + 3 * NSC + 2 * 2 + 1 + 2 * 2 + 2;
  static constexpr int MISC = BAR + NBAR * 8;
  static constexpr int BYTES = MISC + 64;
  static constexpr int ALLOC = BYTES + 1024;             // slack for 1024-byte alignment
  static_assert(SC_BYTES % 128 == 0, "scale stages keep the TMA's 128-byte alignment");
};

// byte offset of the fp16 element (slot k, column n < 64) of a 64-column
// block of the PV B operand: [BN][128 bytes], 128-byte swizzle by slot
__device__ __forceinline__ int mn_elem(int k, int n) { return k * 128 + ((((n >> 3) ^ (k & 7))) << 4) + (n & 7) * 2; }

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
                         const __grid_constant__ CUtensorMap tmQ, RingView rv, int n_q, void* __restrict__ out,
                         int out_f32) {
  using LY = AttnLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived by offsetting the __shared__ array itself
  // so the compiler keeps every access below in the shared address space
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LY::BAR);
  uint64_t* kv_full = bars;                     // [NSTAGE] K, V codes landed
  uint64_t* kv_empty = kv_full + NSTAGE;        // [NSTAGE] K read by QK, V widened
  uint64_t* sc_full = kv_empty + NSTAGE;        // [NSC] raw scales landed
  uint64_t* sc_ready = sc_full + NSC;           // [NSC] scales in the softmax's order (and w) written
  uint64_t* sc_empty = sc_ready + NSC;          // [NSC] the tile's softmax and u columns are done
  uint64_t* s_full = sc_empty + NSC;            // [2] QK done into buffer b
  uint64_t* p_full = s_full + 2;                // [2] every softmax warp has stored its P over buffer b
  uint64_t* pv_done = p_full + 2;               // PV (and row sums) done (once per tile)
  uint64_t* vh_full = pv_done + 1;              // [2] fp16 B operand b written
  uint64_t* vh_free = vh_full + 2;              // [2] PV of the tile in B operand b done
  uint64_t* q_full = vh_free + 2;               // query tile landed
  uint64_t* mma_drain = q_full + 1;             // every issued MMA done (O final; before TMEM is released)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LY::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY::MISC + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int qt = blockIdx.x;
  const int h = blockIdx.y;
  const int H = rv.H;

  if (tid == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1 + CONV_WARPS);   // QK commit, the widening warps
    }
    for (int i = 0; i < NSC; ++i) {
      mbar_init(&sc_full[i], 1);
      mbar_init(&sc_ready[i], CONV_WARPS);
      mbar_init(&sc_empty[i], SOFT_WARPS + CONV_WARPS);   // the softmax, the widening warps
    }
    mbar_init(pv_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], SOFT_WARPS);
      mbar_init(&vh_full[i], CONV_WARPS);
      mbar_init(&vh_free[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == WARP_TMA && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmSK);
    tma_prefetch_desc(&tmSV);
    tma_prefetch_desc(&tmQ);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the set-up above touches no global memory; the ring state, the cache and
  // the query scratch come from earlier kernels
  pdl_wait();
  pdl_trigger();
  const int n_valid = rv.state[ST_NVALID];
  const int T = (n_valid + BN - 1) / BN;

  if (n_valid <= 0) {
    // nothing to attend to: zeros, and a flag the host can read
    if (tid < BM) {
      const int qi = qt * BM + tid;
      if (qi < n_q) {
        const int bytes = D * (out_f32 ? 4 : 2);
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + ((size_t)qi * H + h) * bytes);
        for (int i = 0; i < bytes / 16; ++i) o[i] = make_uint4(0, 0, 0, 0);
      }
    }
    if (tid == 0 && qt == 0 && h == 0) atomicOr(&rv.state[ST_ERR], DEVERR_EMPTY);
  } else if (warp < SOFT_WARPS) {
    // ======================================================== softmax
    // Warp (hf, quarter) reads its 16 TMEM lanes in the 16x256b shape: thread
    // t holds rows t/4 (a) and t/4 + 8 (b) of the half and, of each group of
    // 8 columns, columns 2(t%4) and 2(t%4) + 1.  Four threads share a row.
    const int hf = warp >> 2;
    const int quarter = warp & 3;
    const int c4 = lane & 3;
    const int r4 = lane >> 2;
    const uint32_t lanes = (uint32_t)(32 * quarter + 16 * hf) << 16;
    constexpr float kRowC = (D == 128 ? 0.08838834764831845f : 0.125f) * 1.4426950408889634f;
    const float log2cv = rv.head_stat[2 * h];
    float rq[2], m_run[2];
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      // rows past n_q may hold codes of an earlier call (their output is not
      // stored): a vanishing row factor keeps their logits near zero
      const int qrow = qt * BM + 32 * quarter + 16 * hf + r4 + 8 * sb;
      const float sq = qrow < n_q ? rv.q_scale[(size_t)h * rv.Q_pad + qrow] : 0.0f;
      rq[sb] = sq > 0.0f ? sq * kRowC : 0x1p-100f;
      m_run[sb] = -INFINITY;
    }
    // O and L hold rows weighted by exp2(-m_run): when the running maxima of
    // rows a and b are raised by a tile, the tile's weights use the new
    // maxima at once, and O and L are brought over (times al0, al1) just
    // before the tile's P is stored: once PV_{j-1} (and so every earlier PV)
    // is done, and before PV_j adds the tile.
    auto rescale_o = [&](float al0, float al1) {
      // O's D columns and the 16 of L (the columns past them are unused)
#pragma unroll 1
      for (int c0 = 0; c0 < D + UN; c0 += 32) {
        uint32_t o[16];
        tmem_ld_16x256b_x4(tmem + lanes + TM_O + c0, o);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          o[4 * k] = __float_as_uint(__uint_as_float(o[4 * k]) * al0);
          o[4 * k + 1] = __float_as_uint(__uint_as_float(o[4 * k + 1]) * al0);
          o[4 * k + 2] = __float_as_uint(__uint_as_float(o[4 * k + 2]) * al1);
          o[4 * k + 3] = __float_as_uint(__uint_as_float(o[4 * k + 3]) * al1);
        }
        tmem_st_16x256b_x4(tmem + lanes + TM_O + c0, o);
      }
    };
    bool ok = true;
    for (int j = 0; ok && j < T; ++j) {
      const int b = j & 1;
      const int sc = j % NSC;
      if (!warp_wait(&sc_ready[sc], (j / NSC) & 1, abort_flag) || !warp_wait(&s_full[b], (j >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t xr[64];
      tmem_ld_16x256b_x16(tmem + lanes + TM_S + 128 * b, xr);
      float* x = reinterpret_cast<float*>(xr);
      const uint8_t* stage = sm + LY::SC0 + sc * LY::SC_BYTES;
      const float4* psk = reinterpret_cast<const float4*>(stage + 2 * BN * 4) + c4 * (kPermStride / 4);
      const float4* pw = psk + 4 * (kPermStride / 4);
      const int valid = min(BN, n_valid - j * BN);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // scales of columns 16 i + 2 c4 + {0, 1} and 16 i + 8 + 2 c4 + {0, 1}
        const float4 sk = psk[i];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = 2 * i + e;
          const float2 skp = e ? make_float2(sk.z, sk.w) : make_float2(sk.x, sk.y);
          const float2 ta = mul2(make_float2(x[4 * kk], x[4 * kk + 1]), skp);
          const float2 tb = mul2(make_float2(x[4 * kk + 2], x[4 * kk + 3]), skp);
          x[4 * kk] = ta.x;
          x[4 * kk + 1] = ta.y;
          x[4 * kk + 2] = tb.x;
          x[4 * kk + 3] = tb.y;
        }
      }
      if (valid < BN) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (8 * kk + 2 * c4 + (i & 1) >= valid) x[4 * kk + i] = -INFINITY;
      }
      // maxima of rows a and b over this thread's columns (times the row factor)
      float ma, mb;
      {
        float pa[8], pb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pa[i] = max3f(x[8 * i], x[8 * i + 1], fmaxf(x[8 * i + 4], x[8 * i + 5]));
          pb[i] = max3f(x[8 * i + 2], x[8 * i + 3], fmaxf(x[8 * i + 6], x[8 * i + 7]));
        }
        ma = max3f(max3f(pa[0], pa[1], pa[2]), max3f(pa[3], pa[4], pa[5]), fmaxf(pa[6], pa[7])) * rq[0];
        mb = max3f(max3f(pb[0], pb[1], pb[2]), max3f(pb[3], pb[4], pb[5]), fmaxf(pb[6], pb[7])) * rq[1];
      }
      // The weights use the running maximum of the earlier tiles unless a row
      // of the tile exceeds it by more than the bound (each thread compares
      // the maximum of its own columns, which exceeds the bound whenever the
      // row's does), or on the first tile: then the rows' maxima are formed
      // and raised before the exponentials (O and L follow at the P store).
      float al0 = 1.0f, al1 = 1.0f;
      bool rescale = false;   // warp-uniform
      if (j == 0 || __any_sync(0xFFFFFFFFu, ma > m_run[0] + kLazyRescale || mb > m_run[1] + kLazyRescale)) {
        ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 1));
        mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
        ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 2));
        mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
        const float mn0 = (j == 0 || ma > m_run[0] + kLazyRescale) ? fmaxf(m_run[0], ma + kHeadroom) : m_run[0];
        const float mn1 = (j == 0 || mb > m_run[1] + kLazyRescale) ? fmaxf(m_run[1], mb + kHeadroom) : m_run[1];
        if (j > 0) {
          al0 = ex2f(m_run[0] - mn0);
          al1 = ex2f(m_run[1] - mn1);
          rescale = true;
        }
        m_run[0] = mn0;
        m_run[1] = mn1;
      }
      // weights e = exp2(t * rq + c - m) <= 2^(kLazyLog2 + c)
      {
        const float2 rqa = make_float2(rq[0], rq[0]);
        const float2 rqb = make_float2(rq[1], rq[1]);
        const float2 moa = make_float2(log2cv - m_run[0], log2cv - m_run[0]);
        const float2 mob = make_float2(log2cv - m_run[1], log2cv - m_run[1]);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const float2 aa = fma2(make_float2(x[4 * kk], x[4 * kk + 1]), rqa, moa);
          const float2 ab = fma2(make_float2(x[4 * kk + 2], x[4 * kk + 3]), rqb, mob);
          x[4 * kk] = aa.x;
          x[4 * kk + 1] = aa.y;
          x[4 * kk + 2] = ab.x;
          x[4 * kk + 3] = ab.y;
        }
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) x[i] = ex2f(x[i]);
      // P = e * w in fp16 pairs; the pair of row a at repetition kk goes to
      // P column 4 kk + t%4 of row a (slots 8 kk + 2 t%4 + {0, 1})
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 w4 = pw[i];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = 2 * i + e;
          const float2 wp = e ? make_float2(w4.z, w4.w) : make_float2(w4.x, w4.y);
          const float2 pa2 = mul2(make_float2(x[4 * kk], x[4 * kk + 1]), wp);
          const float2 pb2 = mul2(make_float2(x[4 * kk + 2], x[4 * kk + 3]), wp);
          pk[2 * kk] = cvt_f16x2(pa2.x, pa2.y);
          pk[2 * kk + 1] = cvt_f16x2(pb2.x, pb2.y);
        }
      }
      if (rescale) {
        // PV_{j-2} is done (QK_j, which wrote S_j, was issued after it), so
        // the phase of pv_done that completes next, or last, is PV_{j-1}'s
        if (!warp_wait(pv_done, (j - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        rescale_o(al0, al1);
      }
      // P_j over the S_j just read (this warp's lanes, columns 0 .. 63)
      tmem_st_16x128b_x16(tmem + lanes + TM_S + 128 * b, pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_full[b]);
        mbar_arrive(&sc_empty[sc]);
      }
    }
    // ======================================================== output
    // Both warps of a lane quarter read the row sums of its 32 rows, one row
    // per thread (thread t <-> lane 32*quarter + t), and each writes half of
    // the output columns.
    const int r = 32 * quarter + lane;
    // O and L are final once every MMA is done (after an abort the drain
    // completes too, but the output is then not written)
    ok = ok && warp_wait(mma_drain, 0, abort_flag);
    ok = ok && __shfl_sync(0xFFFFFFFFu, *abort_flag == 0, 0);
    if (ok) {
      tc_fence_after();
      uint32_t lr[2];
      tmem_ld_32x32b_x2(tmem + ((uint32_t)(32 * quarter) << 16) + TM_O + D, lr);
      const float L = __uint_as_float(lr[0]) + __uint_as_float(lr[1]) * 0x1p-11f;
      const float inv_l = 1.0f / ldexpf(L, (int)log2cv);
      const int qi = qt * BM + r;
      const uint32_t row_o = tmem + ((uint32_t)(32 * quarter) << 16) + TM_O;
      uint8_t* orow = static_cast<uint8_t*>(out) + ((size_t)qi * H + h) * (size_t)D * (out_f32 ? 4 : 2);
#pragma unroll 1
      for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
        uint32_t o0[16], o1[16];
        tmem_ld2_32x32b_x16(row_o + c0, row_o + c0 + 16, o0, o1);
        float v[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          v[i] = __uint_as_float(o0[i]) * inv_l;
          v[16 + i] = __uint_as_float(o1[i]) * inv_l;
        }
        if (qi < n_q) {
          if (out_f32) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 4);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                  __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
          } else {
            uint32_t pb[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const __nv_bfloat162 v2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
              pb[i] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 2);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pb[4 * i], pb[4 * i + 1], pb[4 * i + 2], pb[4 * i + 3]);
          }
        }
      }
    }
    tc_fence_before();
  } else if (warp < WARP_TMA) {
    // ======================================================== scales, u columns, V widening
    const int ct = tid - SOFT_THREADS;   // slot ct of every tile
    // the u block of both B operands: columns 2 .. 15 stay zero, columns 0
    // and 1 are written per tile (the rest is never read)
    for (int i = ct; i < 2 * BN * 128 / 16; i += CONV_THREADS)
      reinterpret_cast<uint4*>(sm + LY::VH0 + (i / (BN * 8)) * LY::VH_BYTES + (D / 64) * BN * 128)[i % (BN * 8)] =
          make_uint4(0, 0, 0, 0);
    const float log2cv = rv.head_stat[2 * h];
    const float sfloor = rv.head_stat[2 * h + 1];
    const float cscale = ldexpf(1.0f, -(int)log2cv);   // 2^-c
    // slot ct's place in the softmax's order
    const int ppos = ((ct & 7) >> 1) * kPermStride + 2 * (ct >> 3) + (ct & 1);

    constexpr int CH = D / 16;  // 16-byte e4m3 chunks per slot row
    // Slot ct of tile u: s_k and w = max(s_v, floor) in the softmax's order,
    // and u = 2^-c / w as fp16 u_hi + u_lo * 2^-11 (returned, written into
    // the B operand with the tile's V).  Returns false if the wait gave up.
    auto prep_scales = [&](int u, __half2& uq) -> bool {
      const int sc = u % NSC;
      if (!warp_wait(&sc_full[sc], (u / NSC) & 1, abort_flag)) return false;
      uint8_t* stage = sm + LY::SC0 + sc * LY::SC_BYTES;
      const float sk = reinterpret_cast<const float*>(stage)[ct];
      const float w = fmaxf(reinterpret_cast<const float*>(stage)[BN + ct], sfloor);
      reinterpret_cast<float*>(stage + 2 * BN * 4)[ppos] = sk;
      reinterpret_cast<float*>(stage + 2 * BN * 4)[4 * kPermStride + ppos] = w;
      const float uv = __fdiv_rn(cscale, w);
      const __half uhi = __float2half_rn(uv);
      uq = __halves2half2(uhi, __float2half_rn((uv - __half2float(uhi)) * 2048.0f));
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sc_ready[sc]);
        mbar_arrive(&sc_empty[sc]);
      }
      return true;
    };
    // The scales run two tiles ahead of the widening, so that the softmax of
    // tile u + 1 never waits for the widening of tile u.
    __half2 uq0, uq1, uq2;
    bool ok = prep_scales(0, uq0) && (T < 2 || prep_scales(1, uq1));
    for (int u = 0; ok && u < T; ++u) {
      const int st = u % NSTAGE;
      const int b = u & 1;
      if (u + 2 < T && !prep_scales(u + 2, uq2)) break;
      if (!warp_wait(&kv_full[st], (u / NSTAGE) & 1, abort_flag)) break;
      // B operand b is free once PV_{u-2} is done
      if (u >= 2 && !warp_wait(&vh_free[b], ((u - 2) >> 1) & 1, abort_flag)) break;
      const uint8_t* vsrc = sm + LY::V0 + st * BN * D;
      uint8_t* vdst = sm + LY::VH0 + b * LY::VH_BYTES;
      {
        uint8_t* ub = vdst + (D / 64) * BN * 128;
        *reinterpret_cast<__half2*>(ub + mn_elem(ct, 0)) = uq0;
      }
      // eight consecutive threads take the same chunk of eight consecutive
      // slots, so their 16-byte reads and writes fall in distinct bank groups
#pragma unroll
      for (int it = 0; it < BN * CH / CONV_THREADS; ++it) {
        const int task = it * CONV_THREADS + ct;
        const int sl = 8 * (task / (8 * CH)) + (task & 7);
        const int c = (task >> 3) % CH;
        const uint4 wd = *reinterpret_cast<const uint4*>(vsrc + kmajor_chunk<D>(sl, c));
        uint4 o0, o1;
        o0.x = cvt_e4m3x2_to_f16x2((uint16_t)(wd.x & 0xFFFFu));
        o0.y = cvt_e4m3x2_to_f16x2((uint16_t)(wd.x >> 16));
        o0.z = cvt_e4m3x2_to_f16x2((uint16_t)(wd.y & 0xFFFFu));
        o0.w = cvt_e4m3x2_to_f16x2((uint16_t)(wd.y >> 16));
        o1.x = cvt_e4m3x2_to_f16x2((uint16_t)(wd.z & 0xFFFFu));
        o1.y = cvt_e4m3x2_to_f16x2((uint16_t)(wd.z >> 16));
        o1.z = cvt_e4m3x2_to_f16x2((uint16_t)(wd.w & 0xFFFFu));
        o1.w = cvt_e4m3x2_to_f16x2((uint16_t)(wd.w >> 16));
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
        mbar_arrive(&kv_empty[st]);
      }
      uq0 = uq1;
      uq1 = uq2;
    }
  } else if (warp == WARP_TMA) {
    // ======================================================== TMA producer
    // One lane issues the query tile, then K, V codes into NSTAGE stages and
    // their scales into NSC stages, each as soon as its stage is free: it
    // polls both without blocking (the scales run ahead of the K, V stages)
    // and sleeps briefly when neither can move.  Bounded like every wait.
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, BM * D);
      tma_load_3d(sm + LY::Q, &tmQ, q_full, 0, h, qt * BM);
      int ukv = 0, usc = 0;
      unsigned long long t_last = globaltimer_ns();
      while (ukv < T || usc < T) {
        bool moved = false;
        if (ukv < T && (ukv < NSTAGE || mbar_test_wait(&kv_empty[ukv % NSTAGE], ((ukv / NSTAGE) - 1) & 1))) {
          const int st = ukv % NSTAGE;
          mbar_arrive_expect_tx(&kv_full[st], 2 * BN * D);
          tma_load_3d(sm + LY::K0 + st * BN * D, &tmK, &kv_full[st], 0, ukv * BN, h);
          tma_load_3d(sm + LY::V0 + st * BN * D, &tmV, &kv_full[st], 0, ukv * BN, h);
          ++ukv;
          moved = true;
        }
        if (usc < T && (usc < NSC || mbar_test_wait(&sc_empty[usc % NSC], ((usc / NSC) - 1) & 1))) {
          const int sc = usc % NSC;
          uint8_t* stage = sm + LY::SC0 + sc * LY::SC_BYTES;
          mbar_arrive_expect_tx(&sc_full[sc], 2 * BN * 4);
          tma_load_2d(stage, &tmSK, &sc_full[sc], usc * BN, h);
          tma_load_2d(stage + BN * 4, &tmSV, &sc_full[sc], usc * BN, h);
          ++usc;
          moved = true;
        }
        if (moved) {
          t_last = globaltimer_ns();
        } else {
          if (*abort_flag) break;
          if (globaltimer_ns() - t_last > kWaitLimitNs) {
            *abort_flag = 1;
            break;
          }
          __nanosleep(64);
        }
      }
      if (*abort_flag) {
        // after an abort: let the copies still in flight land in this
        // block's shared memory before the block exits (time-bounded)
        mbar_wait(q_full, 0, nullptr, 100000000ull);
        for (int u = max(0, ukv - NSTAGE); u < ukv; ++u)
          mbar_wait(&kv_full[u % NSTAGE], (u / NSTAGE) & 1, nullptr, 100000000ull);
        for (int u = max(0, usc - NSC); u < usc; ++u)
          mbar_wait(&sc_full[u % NSC], (u / NSC) & 1, nullptr, 100000000ull);
      }
    }
  } else {
    // ======================================================== MMA issue
    // QK_0, QK_1, then per tile j: PV_j (with the row sums) once P_j and the
    // fp16 B operand are in, and QK_{j+2} into buffer j % 2 once PV_j has
    // read P_j there (and K_{j+2} is in).
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc(0, 0, 0, 0, BM, BN);        // e4m3 x e4m3, both K-major
      constexpr uint32_t idesc_pv = make_idesc(0, 0, 0, 1, BM, D + UN);    // f16 x f16, B MN-major
      const uint32_t q_addr = smem_u32(sm + LY::Q);
      auto issue_qk = [&](int u) -> bool {
        const int st = u % NSTAGE;
        if (!mbar_wait(&kv_full[st], (u / NSTAGE) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t ka = smem_u32(sm + LY::K0 + st * BN * D);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          mma_f8_ss(tmem + TM_S + 128 * (u & 1), kmajor_desc<D>(q_addr + kk * 32), kmajor_desc<D>(ka + kk * 32),
                    idesc_qk, kk > 0 ? 1u : 0u);
        mma_commit(&s_full[u & 1]);
        mma_commit(&kv_empty[st]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, abort_flag);
      ok = ok && issue_qk(0);
      if (T > 1) ok = ok && issue_qk(1);
      for (int j = 0; ok && j < T; ++j) {
        const int b = j & 1;
        if (!mbar_wait(&p_full[b], (j >> 1) & 1, abort_flag) || !mbar_wait(&vh_full[b], (j >> 1) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t va = smem_u32(sm + LY::VH0 + b * LY::VH_BYTES);
        // 16 slots per MMA: A = 8 columns of P (fp16 pairs), B = 16 rows of
        // [V | u] (2 KB down the 128-byte rows of each column block)
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_f16_ts(tmem + TM_O, tmem + TM_S + 128 * b + kk * 8, make_sdesc_sw128(va + kk * 16 * 128, BN * 128, 1024),
                     idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(pv_done);
        mma_commit(&vh_free[b]);
        if (j + 2 < T) {
          // QK_{j+2} overwrites the P that PV_j reads
          if (!mbar_wait(pv_done, j & 1, abort_flag)) break;
          tc_fence_after();
          if (!issue_qk(j + 2)) break;
        }
      }
      // every MMA issued so far is done before the block releases TMEM
      mma_commit(mma_drain);
      mbar_wait(mma_drain, 0, nullptr, 100000000ull);
    }
  }

  __syncthreads();
  if (tid == 0 && *abort_flag) atomicOr(&rv.state[ST_ERR], DEVERR_TIMEOUT);
  if (warp == WARP_MMA) {
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

cudaError_t launch_fp8_ring_attn(const RingView& rv, const AttnMaps& maps, const CUtensorMap& tmQ, int n_q, void* out,
                                 int out_f32, cudaStream_t st) {
  const dim3 grid((n_q + BM - 1) / BM, rv.H);
  if (rv.D == 128)
    return launch_pdl(fp8_ring_attn_kernel<128>, grid, dim3(ATT_THREADS), AttnLayout<128>::ALLOC, st, maps.k_codes,
                      maps.v_codes, maps.k_scale, maps.v_scale, tmQ, rv, n_q, out, out_f32);
  return launch_pdl(fp8_ring_attn_kernel<64>, grid, dim3(ATT_THREADS), AttnLayout<64>::ALLOC, st, maps.k_codes,
                    maps.v_codes, maps.k_scale, maps.v_scale, tmQ, rv, n_q, out, out_f32);
}

}  // namespace kvring_dev
