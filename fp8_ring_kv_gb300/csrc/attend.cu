// fp8_ring_attn: n_q queries attend over every valid slot of the FP8 ring.
//
// Runway Characters paper, §4.3 (K and V stored as float8_e4m3, the queries
// quantised per call, attention reading the FP8 cache directly) and
// Appendix G (each call reads all the cache's slots; no causal mask).
//
// The queries arrive rotated and e4m3-coded, with one scale per (query,
// head), from the query preparation kernel (query scratch of the workspace).
// One block per (tile of 128 queries, head).  The slots are visited in tiles
// of 128 in storage order: attention is a sum over the valid slots, so the
// ring's wrap needs no reordering, and slots >= n_valid are masked.
//
//   S_j  = Qcodes . Kcodes_j^T            tcgen05 kind::f8f6f4, fp32 in TMEM
//   t    = S_j * s_k (per column);  logit*log2(e) = t * s_q * log2(e)/sqrt(D)
//   online softmax in base 2: e = exp2(t*r - m + c), with a running row
//   maximum m that is only raised (and O, L rescaled) when a tile's maximum
//   exceeds it by more than 2^14, so e <= 2^14 * 2^c
//   P_j  = e * w (per column, w = max(s_v, floor)) rounded to fp16, in TMEM
//   O   += P_j . Vcodes_j                  tcgen05 kind::f16 (A = P from TMEM)
//   L   += P_j . [u_hi | u_lo]_j           the same, N = 16: u = 2^-c / w
//   out  = O / (L * 2^c)
// The e4m3 V codes are widened to fp16 in shared memory (exact) because the
// fp16 MMA takes both operands in fp16; P in fp16 keeps the weighted sum of V
// within the accuracy that e4m3 weights would lose.  2^c is a per-head power of
// two (cancelling between O and L) that keeps P within fp16 range.
//
// The row sums L are taken from the same fp16 P as the weighted sum of V (u
// split into two fp16 parts, u_hi + u_lo * 2^-11, good to about 2^-22), so the
// rounding of each P cancels between O and L: a row dominated by one slot
// returns that slot's value, not the value times the fp16 rounding of its
// weight (up to 2^-11 of |v|).  The per-head floor, 2^-15 * max(max s_v,
// 2^-c), keeps a zero or near-zero V row's weight in L; it changes that row's
// own (near-zero) values by at most 448 * floor.
//
// Pipeline.  S has two TMEM buffers (2 x 128 columns), P one (64), then L (16
// of 32 columns) and O (D).  The MMA sequence is QK_0, QK_1, QK_2, PV_0, QK_3,
// PV_1, ...: while the softmax works on tile j the tensor cores run QK_{j+1}
// and PV_{j-1} (with its row sums), and each MMA waits only for the softmax of
// the tile it consumes or frees; the softmax of tile j stores its P once
// PV_{j-1} has read the previous one.  TMEM lane quarter q can only be read by the warps of SM
// sub-partition q, so the softmax of rows 32q .. 32q+31 runs on one
// sub-partition and its per-tile cost sets the pace.
//
// Warp roles (448 threads):
//   warps 0-7   softmax: warp w serves the 16-lane half w/4 of TMEM lane
//               quarter w%4; finally the output, half of the columns each
//   warps 8-11  the per-head fp16 range factor and scale floor, then per
//               tile the widening of V to fp16 and the u columns (one warp
//               per SM sub-partition)
//   warp 12     TMA producer (the e4m3 query tile, then K, V codes into 4
//               stages and their scales into 8)
//   warp 13     TMEM allocation and MMA issue
// The softmax and MMA warps poll their barriers; the TMA and widening warps,
// whose work runs ahead of need, park while they wait so that their polling
// does not take issue slots from the softmax warps beside them.
#include <cfloat>

#include "common.cuh"
#include "launch.h"

namespace kvring_dev {

constexpr int BM = 128;           // query rows per block
constexpr int BN = 128;           // slots per tile
constexpr int NSTAGE = 4;         // fp8 K/V stages
constexpr int NSC = 8;            // scale stages (held until the tile's softmax ends)
constexpr int ATT_THREADS = 448;
constexpr int SOFT_WARPS = 8;
constexpr int SOFT_THREADS = 32 * SOFT_WARPS;
constexpr int CONV_WARPS = 4;
constexpr int CONV_THREADS = 32 * CONV_WARPS;
constexpr int WARP_TMA = SOFT_WARPS + CONV_WARPS;
constexpr int WARP_MMA = WARP_TMA + 1;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;      // S buffer b: fp32 [128 lanes][128] at columns 128 b
constexpr uint32_t TM_P = 256;    // P: fp16 pairs [128 lanes][64]
constexpr uint32_t TM_L = 352;    // L: fp32 [128 lanes][16] (columns 0, 1: hi and lo sums) of 32 kept
constexpr uint32_t TM_O = 384;    // O: fp32 [128 lanes][D], right after L's 32 columns
constexpr int UN = 16;            // columns of the row-sum MMA
// log2 of the scale floor under the head's largest V scale (and of the
// largest u, which must stay inside fp16)
constexpr int kFloorLog2 = 15;
// log2 of the largest unnormalised weight.  A wider bound makes rescales (a
// wait for the previous PV, O and L rescaled) rarer, but the per-head factor
// 2^c that keeps every P = weight * w * 2^c below fp16's maximum then puts
// the row's largest P lower, and more of its small weights into fp16
// subnormals or zero.  Those weights are lost to L as well as to O, and with
// many of them that changes the output.  Right after a row's maximum is set,
// its largest P is 2^(14 - kLazyLog2 - kHeadroom) = 2^0 (times w 2^c in
// [1, 2)), so weights down to 2^-14 of it stay normal.
constexpr int kLazyLog2 = 10;
constexpr float kLazyRescale = (float)kLazyLog2;
// A running maximum is set this many octaves above the tile maximum that sets
// it (weights then start at most 2^-4), so later tiles may exceed the observed
// maximum by kLazyLog2 + 4 octaves before a rescale.
constexpr float kHeadroom = 4.0f;

template <int D>
struct AttnLayout {
  static constexpr int Q = 0;                            // e4m3 [BM][D], K-major swizzled
  static constexpr int K0 = Q + BM * D;                  // NSTAGE x e4m3 [BN][D]
  static constexpr int V0 = K0 + NSTAGE * BN * D;        // NSTAGE x e4m3 [BN][D]
  static constexpr int VH0 = V0 + NSTAGE * BN * D;       // 2 x fp16 [BN][D], MN-major swizzled
  static constexpr int U0 = VH0 + 2 * BN * D * 2;        // 2 x fp16 [UN][BN], K-major, 128-byte swizzle
  static constexpr int SC0 = U0 + 2 * UN * BN * 2;       // NSC x fp32 {s_k [BN], s_v [BN]}
  static constexpr int BAR = SC0 + NSC * 2 * BN * 4;
  static constexpr int NBAR = 2 * NSTAGE + 2 * NSC + 9;
  static constexpr int MISC = BAR + NBAR * 8;
  static constexpr int BYTES = MISC + 64;
  static constexpr int ALLOC = BYTES + 1024;             // slack for 1024-byte alignment
};

// byte offset of the fp16 element (row n, slot k) of a u tile: two 64-slot
// atoms of [UN rows][128 bytes], 128-byte swizzle
__device__ __forceinline__ int u_elem(int n, int k) {
  return (k >> 6) * (UN * 128) + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2;
}

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
  uint64_t* sc_full = kv_empty + NSTAGE;        // [NSC] scales landed
  uint64_t* sc_empty = sc_full + NSC;           // [NSC] the tile's softmax and u columns are done
  uint64_t* s_full = sc_empty + NSC;            // [2] QK done into S buffer b
  uint64_t* p_full = s_full + 2;                // [2] P of tile parity b stored, S buffer b read
  uint64_t* pv_done = p_full + 2;               // [2] PV and row sums of tile parity b done
  uint64_t* vh_full = pv_done + 2;              // [2] fp16 V buffer b and u tile b written
  uint64_t* q_full = vh_full + 2;               // query tile + range factor
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LY::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY::MISC + 4);
  int* maxsv_bits = reinterpret_cast<int*>(sm + LY::MISC + 8);
  float* cv_smem = reinterpret_cast<float*>(sm + LY::MISC + 12);   // log2 of the per-head weight factor
  float* floor_smem = reinterpret_cast<float*>(sm + LY::MISC + 16);  // the per-head scale floor

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
      mbar_init(&sc_empty[i], SOFT_WARPS + CONV_WARPS);   // the softmax, the u columns
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], SOFT_WARPS);
      mbar_init(&pv_done[i], 1);
      mbar_init(&vh_full[i], CONV_WARPS);
    }
    mbar_init(q_full, 1 + CONV_WARPS);   // the query tile's TMA, the widening warps (range factor)
    *abort_flag = 0;
    *maxsv_bits = 0;
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
    // 8 columns, columns 2(t%4) and 2(t%4) + 1.  Four threads share a row and
    // each needs only its 32 columns' scales.
    const int hf = warp >> 2;
    const int quarter = warp & 3;
    const int c4 = lane & 3;
    const int r4 = lane >> 2;
    const uint32_t lanes = (uint32_t)(32 * quarter + 16 * hf) << 16;
    const uint32_t lo_addr = tmem + lanes + TM_L;   // L's 32 columns, then O
    constexpr float kRowC = (D == 128 ? 0.08838834764831845f : 0.125f) * 1.4426950408889634f;
    float rq[2], m_run[2];
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      const int qrow = qt * BM + 32 * quarter + 16 * hf + r4 + 8 * sb;
      const float sq = qrow < n_q ? rv.q_scale[(size_t)h * rv.Q_pad + qrow] : 0.0f;
      rq[sb] = sq > 0.0f ? sq * kRowC : 1.0f;
      m_run[sb] = -INFINITY;
    }
    bool ok = mbar_wait(q_full, 0, abort_flag);
    const float log2cv = *cv_smem;
    const float sfloor = *floor_smem;
    // Raise the running maxima of rows a and b to mn0, mn1 at tile j > 0:
    // O and L hold rows weighted by exp2(-m_run), so once PV_{j-1} (and so
    // every earlier PV and row sum) is done they are brought to exp2(-m_new).
    // Returns the factors 2^(m_old - m_new); false if the wait gave up.
    auto raise_max = [&](int j, float mn0, float mn1, float& al0, float& al1) -> bool {
      al0 = 1.0f;
      al1 = 1.0f;
      if (j > 0) {
        if (!mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        al0 = ex2f(m_run[0] - mn0);
        al1 = ex2f(m_run[1] - mn1);
#pragma unroll 1
        for (int c0 = 0; c0 < 32 + D; c0 += 32) {
          uint32_t o[16];
          tmem_ld_16x256b_x4(lo_addr + c0, o);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            o[4 * k] = __float_as_uint(__uint_as_float(o[4 * k]) * al0);
            o[4 * k + 1] = __float_as_uint(__uint_as_float(o[4 * k + 1]) * al0);
            o[4 * k + 2] = __float_as_uint(__uint_as_float(o[4 * k + 2]) * al1);
            o[4 * k + 3] = __float_as_uint(__uint_as_float(o[4 * k + 3]) * al1);
          }
          tmem_st_16x256b_x4(lo_addr + c0, o);
        }
      }
      m_run[0] = mn0;
      m_run[1] = mn1;
      return true;
    };
    for (int j = 0; ok && j < T; ++j) {
      const int b = j & 1;
      const int sc = j % NSC;
      if (!mbar_wait(&sc_full[sc], (j / NSC) & 1, abort_flag) || !mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = tmem + lanes + TM_S + 128 * b;
      // column 8k + 2*c4 of the tile's scales at [8k]
      const float* skp = reinterpret_cast<const float*>(sm + LY::SC0 + sc * 2 * BN * 4) + 2 * c4;
      const float* svp = skp + BN;
      const int valid = min(BN, n_valid - j * BN);
      // The weights use the running maximum from the earlier tiles while the
      // tile's own maximum is found alongside; each thread compares the
      // maximum of its own columns, which exceeds the bound whenever the
      // row's does.  Only then (and always on the first tile) is the row
      // maximum formed, raised, O and the sums rescaled, and the tile
      // recomputed from S, which stays in TMEM until this tile's end.
      uint32_t pk[32];
      for (int pass = (j == 0 ? 1 : 0); pass < 2; ++pass) {
        uint32_t xr[64];
        tmem_ld_16x256b_x16(s_addr, xr);
        float* x = reinterpret_cast<float*>(xr);
        {
          float2 sk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) sk[k] = *reinterpret_cast<const float2*>(skp + 8 * k);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 ta = mul2(make_float2(x[4 * k], x[4 * k + 1]), sk[k]);
            const float2 tb = mul2(make_float2(x[4 * k + 2], x[4 * k + 3]), sk[k]);
            x[4 * k] = ta.x;
            x[4 * k + 1] = ta.y;
            x[4 * k + 2] = tb.x;
            x[4 * k + 3] = tb.y;
          }
        }
        if (valid < BN) {
#pragma unroll
          for (int k = 0; k < 16; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (8 * k + 2 * c4 + (i & 1) >= valid) x[4 * k + i] = -INFINITY;
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
        if (pass == 1) {
          // row maxima over the four threads of each row
          ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 1));
          mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
          ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 2));
          mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
          const bool grow0 = j == 0 || ma > m_run[0] + kLazyRescale;
          const bool grow1 = j == 0 || mb > m_run[1] + kLazyRescale;
          const float mn0 = grow0 ? fmaxf(m_run[0], ma + kHeadroom) : m_run[0];
          const float mn1 = grow1 ? fmaxf(m_run[1], mb + kHeadroom) : m_run[1];
          float al0, al1;
          if (!raise_max(j, mn0, mn1, al0, al1)) {
            ok = false;
            break;
          }
        }
        // weights e = exp2(t * rq + c - m), P = e * s_v in fp16 pairs; the
        // pair of row a at repetition k goes to P column 4k + t%4 of row a
        const float2 rqa = make_float2(rq[0], rq[0]);
        const float2 rqb = make_float2(rq[1], rq[1]);
        const float2 moa = make_float2(log2cv - m_run[0], log2cv - m_run[0]);
        const float2 mob = make_float2(log2cv - m_run[1], log2cv - m_run[1]);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 aa = fma2(make_float2(x[4 * k], x[4 * k + 1]), rqa, moa);
          const float2 ab = fma2(make_float2(x[4 * k + 2], x[4 * k + 3]), rqb, mob);
          x[4 * k] = aa.x;
          x[4 * k + 1] = aa.y;
          x[4 * k + 2] = ab.x;
          x[4 * k + 3] = ab.y;
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = ex2f(x[i]);
        // A row whose tile maximum passed the bound (decided only now, so that
        // the maxima overlap the exponentials): raise its maximum and scale the
        // weights just computed, in fp32, by 2^(m_old - m_new) -- the same as
        // recomputing them up to rounding -- unless one of them overflowed,
        // in which case the tile is recomputed from S (pass 1).
        if (pass == 0 && __any_sync(0xFFFFFFFFu, ma > m_run[0] + kLazyRescale || mb > m_run[1] + kLazyRescale)) {
          ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 1));
          mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
          ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 2));
          mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
          bool finite = true;
#pragma unroll
          for (int i = 0; i < 64; ++i) finite = finite && x[i] < INFINITY;
          if (!__all_sync(0xFFFFFFFFu, finite)) continue;   // -> pass 1
          const float mn0 = ma > m_run[0] + kLazyRescale ? ma + kHeadroom : m_run[0];
          const float mn1 = mb > m_run[1] + kLazyRescale ? mb + kHeadroom : m_run[1];
          float al0, al1;
          if (!raise_max(j, mn0, mn1, al0, al1)) {
            ok = false;
            break;
          }
          const float2 fa = make_float2(al0, al0), fb = make_float2(al1, al1);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 ea = mul2(make_float2(x[4 * k], x[4 * k + 1]), fa);
            const float2 eb = mul2(make_float2(x[4 * k + 2], x[4 * k + 3]), fb);
            x[4 * k] = ea.x;
            x[4 * k + 1] = ea.y;
            x[4 * k + 2] = eb.x;
            x[4 * k + 3] = eb.y;
          }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float2 sv = *reinterpret_cast<const float2*>(svp + 8 * k);
          sv.x = fmaxf(sv.x, sfloor);
          sv.y = fmaxf(sv.y, sfloor);
          const float2 pa2 = mul2(make_float2(x[4 * k], x[4 * k + 1]), sv);
          const float2 pb2 = mul2(make_float2(x[4 * k + 2], x[4 * k + 3]), sv);
          pk[2 * k] = cvt_f16x2(pa2.x, pa2.y);
          pk[2 * k + 1] = cvt_f16x2(pb2.x, pb2.y);
        }
        break;
      }
      if (!ok) break;
      // P is free once PV_{j-1} (and its row sums) have read it
      if (j >= 1 && !mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st_16x128b_x16(tmem + lanes + TM_P, pk);
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
    ok = ok && mbar_wait(&pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, abort_flag);
    if (ok) {
      tc_fence_after();
      uint32_t lr[2];
      tmem_ld_32x32b_x2(tmem + ((uint32_t)(32 * quarter) << 16) + TM_L, lr);
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
    // ======================================================== range factor + V widening
    const int ct = tid - SOFT_THREADS;
    {
      // the largest V scale of this head (each head's scale row starts
      // 16-byte aligned: rows are S_pad = S rounded up to 4 apart)
      const float* vs1 = rv.v_scale + (size_t)h * rv.S_pad;
      const float4* vs = reinterpret_cast<const float4*>(vs1);
      const int n4 = n_valid >> 2;
      float mx = 0.0f;
#pragma unroll 4
      for (int i = ct; i < n4; i += CONV_THREADS) {
        const float4 v = __ldg(vs + i);
        mx = fmaxf(mx, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
      }
      if (ct < (n_valid & 3)) mx = fmaxf(mx, vs1[n4 * 4 + ct]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      if (lane == 0) atomicMax(maxsv_bits, __float_as_int(mx));
      asm volatile("bar.sync 1, %0;" ::"n"(CONV_THREADS) : "memory");
      if (ct == 0) {
        const float m = __int_as_float(*maxsv_bits);
        // weights reach 2^kLazyLog2 * 2^c; with c = 14 - kLazyLog2 -
        // floor(log2 max s_v) every P = weight * w stays below 2^15 (fp16
        // max 65504), w = max(s_v, floor) <= max(max s_v, 2^-c)
        int c = m > 0.0f ? 14 - kLazyLog2 - ilogbf(m) : 0;
        c = c < -64 ? -64 : (c > 64 ? 64 : c);
        *cv_smem = (float)c;
        // the scale floor: u = 2^-c / max(s_v, floor) <= 2^kFloorLog2
        *floor_smem = ldexpf(fmaxf(m, ldexpf(1.0f, -c)), -kFloorLog2);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(CONV_THREADS) : "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }

    // u tiles: rows 2 .. UN-1 stay zero; rows 0 and 1 are written per tile
    for (int i = ct; i < 2 * UN * BN * 2 / 16; i += CONV_THREADS)
      reinterpret_cast<uint4*>(sm + LY::U0)[i] = make_uint4(0, 0, 0, 0);
    const float cscale = ldexpf(1.0f, -(int)*cv_smem);   // 2^-c
    const float sfloor = *floor_smem;

    constexpr int CH = D / 16;  // 16-byte e4m3 chunks per slot row
    for (int u = 0; u < T; ++u) {
      const int st = u % NSTAGE;
      const int sc = u % NSC;
      const int b = u & 1;
      if (!mbar_wait<true>(&kv_full[st], (u / NSTAGE) & 1, abort_flag)) break;
      // fp16 V buffer b and u tile b are free once PV_{u-2} is done
      if (u >= 2 && !mbar_wait<true>(&pv_done[b], ((u - 2) >> 1) & 1, abort_flag)) break;
      if (!mbar_wait<true>(&sc_full[sc], (u / NSC) & 1, abort_flag)) break;
      {
        // slot ct of the tile: u = 2^-c / max(s_v, floor) as fp16 u_hi + u_lo * 2^-11
        const float sv = reinterpret_cast<const float*>(sm + LY::SC0 + sc * 2 * BN * 4)[BN + ct];
        const float uv = __fdiv_rn(cscale, fmaxf(sv, sfloor));
        const __half hi = __float2half_rn(uv);
        const __half lo = __float2half_rn((uv - __half2float(hi)) * 2048.0f);
        uint8_t* ut = sm + LY::U0 + b * UN * BN * 2;
        *reinterpret_cast<__half*>(ut + u_elem(0, ct)) = hi;
        *reinterpret_cast<__half*>(ut + u_elem(1, ct)) = lo;
      }
      const uint8_t* vsrc = sm + LY::V0 + st * BN * D;
      uint8_t* vdst = sm + LY::VH0 + b * BN * D * 2;
      // eight consecutive threads take the same chunk of eight consecutive
      // slots, so their 16-byte reads and writes fall in distinct bank groups
#pragma unroll
      for (int it = 0; it < BN * CH / CONV_THREADS; ++it) {
        const int task = it * CONV_THREADS + ct;
        const int sl = 8 * (task / (8 * CH)) + (task & 7);
        const int c = (task >> 3) % CH;
        const uint4 w = *reinterpret_cast<const uint4*>(vsrc + kmajor_chunk<D>(sl, c));
        uint4 o0, o1;
        o0.x = cvt_e4m3x2_to_f16x2((uint16_t)(w.x & 0xFFFFu));
        o0.y = cvt_e4m3x2_to_f16x2((uint16_t)(w.x >> 16));
        o0.z = cvt_e4m3x2_to_f16x2((uint16_t)(w.y & 0xFFFFu));
        o0.w = cvt_e4m3x2_to_f16x2((uint16_t)(w.y >> 16));
        o1.x = cvt_e4m3x2_to_f16x2((uint16_t)(w.z & 0xFFFFu));
        o1.y = cvt_e4m3x2_to_f16x2((uint16_t)(w.z >> 16));
        o1.z = cvt_e4m3x2_to_f16x2((uint16_t)(w.w & 0xFFFFu));
        o1.w = cvt_e4m3x2_to_f16x2((uint16_t)(w.w >> 16));
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
        mbar_arrive(&sc_empty[sc]);
      }
    }
  } else if (warp == WARP_TMA) {
    // ======================================================== TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, BM * D);
      tma_load_3d(sm + LY::Q, &tmQ, q_full, 0, h, qt * BM);
      for (int u = 0; u < T; ++u) {
        const int st = u % NSTAGE;
        const int sc = u % NSC;
        if (u >= NSTAGE && !mbar_wait<true>(&kv_empty[st], ((u / NSTAGE) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * BN * D);
        tma_load_3d(sm + LY::K0 + st * BN * D, &tmK, &kv_full[st], 0, u * BN, h);
        tma_load_3d(sm + LY::V0 + st * BN * D, &tmV, &kv_full[st], 0, u * BN, h);
        if (u >= NSC && !mbar_wait<true>(&sc_empty[sc], ((u / NSC) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(&sc_full[sc], 2 * BN * 4);
        tma_load_2d(sm + LY::SC0 + sc * 2 * BN * 4, &tmSK, &sc_full[sc], u * BN, h);
        tma_load_2d(sm + LY::SC0 + sc * 2 * BN * 4 + BN * 4, &tmSV, &sc_full[sc], u * BN, h);
      }
    }
  } else {
    // ======================================================== MMA issue
    // QK_0, QK_1, then per tile j, once the softmax of tile j is done: QK_{j+2}
    // into the S buffer it has finished reading, then PV_j and its row sums.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc(0, 0, 0, 0, BM, BN);   // e4m3 x e4m3, both K-major
      constexpr uint32_t idesc_pv = make_idesc(0, 0, 0, 1, BM, D);    // f16 x f16, V MN-major
      constexpr uint32_t idesc_l = make_idesc(0, 0, 0, 0, BM, UN);    // f16 x f16, u K-major
      bool ok = mbar_wait(q_full, 0, abort_flag);
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
      ok = ok && issue_qk(0);
      if (T > 1) ok = ok && issue_qk(1);
      for (int j = 0; ok && j < T; ++j) {
        const int b = j & 1;
        if (!mbar_wait(&p_full[b], (j >> 1) & 1, abort_flag) || !mbar_wait(&vh_full[b], (j >> 1) & 1, abort_flag))
          break;
        tc_fence_after();
        if (j + 2 < T && !issue_qk(j + 2)) break;
        const uint32_t va = smem_u32(sm + LY::VH0 + b * BN * D * 2);
        const uint32_t ua = smem_u32(sm + LY::U0 + b * UN * BN * 2);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_f16_ts(tmem + TM_O, tmem + TM_P + kk * 8, make_sdesc_sw128(va + kk * 16 * 128, BN * 128, 1024),
                     idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        // 16 slots (32 bytes) per MMA; four per 64-slot atom
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_f16_ts(tmem + TM_L, tmem + TM_P + kk * 8,
                     make_sdesc_sw128(ua + (kk >> 2) * (UN * 128) + (kk & 3) * 32, 16, 1024), idesc_l,
                     (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&pv_done[b]);
      }
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
