// Host side of libkvring: argument checks, workspace layout, RoPE tables,
// TMA descriptors and kernel launches.  See include/kvring.h for the contract.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/kvring.h"
#include "launch.h"

using namespace kvring_dev;

// Query scratch of kvring_attend_noalloc: one array per device, part of the
// library's device image (no allocation at run time).  Nothing in it has to
// start at zero.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVRING_NOALLOC_SCRATCH_BYTES];

struct kvring {
  kvring_config cfg;
  RingView rv;
  AttnMaps maps;
  CUtensorMap q_map;  // e4m3 query scratch, [max_queries][H][D]
  int device;
  // call order, tracked on the host (the calls are enqueued in host order)
  bool globals_written;
  bool window_written;
  bool calibrated;
};

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return KVRING_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t state, rope[3], k_codes, v_codes, k_scale, v_scale, stat, q_codes, q_scale, head_stat, total;
  int s_pad, q_pad;
};

bool check_config(const kvring_config* c) {
  if (!c) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->heads < 1 || 2 * c->heads * (c->head_dim / 16) > 1024) return false;
  if (c->n_slots < 1 || c->n_slots > (1 << 20)) return false;
  if (c->n_axes < 1 || c->n_axes > 3) return false;
  int sum = 0;
  for (int a = 0; a < c->n_axes; ++a) {
    if (c->axis_dims[a] < 2 || c->axis_dims[a] % 2) return false;
    if (c->pos_count[a] < 1 || c->pos_count[a] > (1 << 24)) return false;
    sum += c->axis_dims[a];
  }
  if (sum != c->head_dim) return false;
  if (!(c->rope_base > 1.0) || !std::isfinite(c->rope_base)) return false;
  if (c->out_dtype != KVRING_OUT_BF16 && c->out_dtype != KVRING_OUT_F32) return false;
  if (c->max_queries < 1 || c->max_queries > (1 << 20)) return false;
  if (c->n_global < 0 || c->n_global >= c->n_slots) return false;
  if (c->scale_mode != KVRING_SCALES_TOKEN && c->scale_mode != KVRING_SCALES_STATIC) return false;
  return true;
}

Layout layout_of(const kvring_config* c) {
  Layout L{};
  const size_t H = c->heads, D = c->head_dim, S = c->n_slots;
  L.s_pad = (int)round_up(S, 4);
  size_t off = 0;
  L.state = off;
  off = round_up(off + ST_WORDS * sizeof(int32_t), 1024);
  for (int a = 0; a < 3; ++a) {
    L.rope[a] = off;
    if (a < c->n_axes) off = round_up(off + (size_t)c->pos_count[a] * (c->axis_dims[a] / 2) * sizeof(float2), 1024);
  }
  L.k_codes = off;
  off = round_up(off + H * S * D, 1024);
  L.v_codes = off;
  off = round_up(off + H * S * D, 1024);
  L.k_scale = off;
  off = round_up(off + H * L.s_pad * sizeof(float), 1024);
  L.v_scale = off;
  off = round_up(off + H * L.s_pad * sizeof(float), 1024);
  L.stat = off;
  off = round_up(off + 6 * H * sizeof(float), 1024);
  L.q_pad = (int)round_up(c->max_queries, 4);
  L.q_codes = off;
  off = round_up(off + (size_t)c->max_queries * H * D, 1024);
  L.q_scale = off;
  off = round_up(off + H * L.q_pad * sizeof(float), 1024);
  L.head_stat = off;
  off = round_up(off + 2 * H * sizeof(float), 1024);
  L.total = off;
  return L;
}

// omega_{a,j} = base^(-2j/d_a), fp64
double omega(double base, int d_axis, int j) { return std::pow(base, -2.0 * j / d_axis); }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Query codes [n_rows][H][D] at q_codes: box of D channels x 1 head x 128
// queries, swizzled like the key tiles (rows beyond n_rows read as zero).
bool encode_query_map(CUtensorMap* m, const void* q_codes, int H, int D, int n_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)n_rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)H * D};
  const cuuint32_t box[3] = {(cuuint32_t)D, 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q_codes), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_maps(kvring* r) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const RingView& rv = r->rv;
  const cuuint64_t D = rv.D, S = rv.S, H = rv.H;
  const CUtensorMapSwizzle sw = rv.D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (!encode_query_map(&r->q_map, rv.q_codes, rv.H, rv.D, r->cfg.max_queries)) return false;
  {
    const cuuint64_t dims[3] = {D, S, H};
    const cuuint64_t strides[2] = {D, S * D};
    const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)kAttnKeyTile, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&r->maps.k_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, rv.k_codes, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
    if (enc(&r->maps.v_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, rv.v_codes, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)rv.S_pad, H};
    const cuuint64_t strides[1] = {(cuuint64_t)rv.S_pad * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kAttnKeyTile, 1};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&r->maps.k_scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, rv.k_scale, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
    if (enc(&r->maps.v_scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, rv.v_scale, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.
constexpr int kNoallocDevices = 64;
std::atomic<uint8_t*> g_noalloc_addr[kNoallocDevices];
std::mutex g_noalloc_setup;

int noalloc_scratch(int dev, uint8_t** out) {
  if (dev < 0 || dev >= kNoallocDevices) return KVRING_ERR_UNSUPPORTED;
  uint8_t* p = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_noalloc_setup);
    p = g_noalloc_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      void* a = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e);
      p = static_cast<uint8_t*>(a);
      g_noalloc_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return KVRING_OK;
}

// cos/sin of the rotation by -d on the temporal axis, fp64 then rounded once
DeltaTable delta_table(const kvring_config& cfg, int32_t d) {
  DeltaTable dt{};
  dt.n_pairs = cfg.axis_dims[0] / 2;
  for (int j = 0; j < dt.n_pairs; ++j) {
    const double th = -(double)d * omega(cfg.rope_base, cfg.axis_dims[0], j);
    dt.cs[j] = make_float2((float)std::cos(th), (float)std::sin(th));
  }
  return dt;
}

}  // namespace

extern "C" {

size_t kvring_workspace_bytes(const kvring_config* cfg) {
  if (!check_config(cfg)) return 0;
  return layout_of(cfg).total;
}

int kvring_create(const kvring_config* cfg, void* workspace, size_t workspace_bytes, kvring_stream stream,
                  kvring** out) {
  if (!out) return KVRING_ERR_INVALID_ARG;
  *out = nullptr;
  if (!check_config(cfg) || !workspace) return KVRING_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return KVRING_ERR_MISALIGNED;
  const Layout L = layout_of(cfg);
  if (workspace_bytes < L.total) return KVRING_ERR_WORKSPACE;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  int major = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (major != 10) return KVRING_ERR_NO_DEVICE;

  kvring* r = new (std::nothrow) kvring;
  if (!r) return KVRING_ERR_INVALID_ARG;
  std::memset(r, 0, sizeof(*r));
  r->cfg = *cfg;
  r->device = dev;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  RingView& rv = r->rv;
  rv.state = reinterpret_cast<int32_t*>(ws + L.state);
  int pair_off = 0;
  for (int a = 0; a < 3; ++a) {
    const bool on = a < cfg->n_axes;
    rv.rope[a] = on ? reinterpret_cast<const float2*>(ws + L.rope[a]) : nullptr;
    rv.pos_min[a] = on ? cfg->pos_min[a] : 0;
    rv.pos_count[a] = on ? cfg->pos_count[a] : 1;
    rv.axis_pairs[a] = on ? cfg->axis_dims[a] / 2 : 0;
    rv.pair_off[a] = pair_off;
    if (on) pair_off += cfg->axis_dims[a] / 2;
  }
  rv.k_codes = ws + L.k_codes;
  rv.v_codes = ws + L.v_codes;
  rv.k_scale = reinterpret_cast<float*>(ws + L.k_scale);
  rv.v_scale = reinterpret_cast<float*>(ws + L.v_scale);
  rv.q_codes = ws + L.q_codes;
  rv.q_scale = reinterpret_cast<float*>(ws + L.q_scale);
  rv.head_stat = reinterpret_cast<float*>(ws + L.head_stat);
  rv.Q_pad = L.q_pad;
  rv.H = cfg->heads;
  rv.D = cfg->head_dim;
  rv.S = cfg->n_slots;
  rv.S_pad = L.s_pad;
  rv.n_axes = cfg->n_axes;
  rv.G = cfg->n_global;
  rv.stat = reinterpret_cast<float*>(ws + L.stat);
  rv.scale_mode = cfg->scale_mode;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // state, codes and scales (and the query scratch) start at zero: an empty ring
  if ((e = cudaMemsetAsync(ws + L.state, 0, L.rope[0] - L.state, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(ws + L.k_codes, 0, L.total - L.k_codes, st)) != cudaSuccess) {
    delete r;
    return cuda_fail(e);
  }
  // RoPE tables: fp32 cos/sin of pos * omega_{a,j}, angle formed in fp64
  for (int a = 0; a < cfg->n_axes; ++a) {
    const int J = cfg->axis_dims[a] / 2;
    std::vector<float2> tab((size_t)cfg->pos_count[a] * J);
    for (int i = 0; i < cfg->pos_count[a]; ++i) {
      const double p = (double)cfg->pos_min[a] + i;
      for (int j = 0; j < J; ++j) {
        const double th = p * omega(cfg->rope_base, cfg->axis_dims[a], j);
        tab[(size_t)i * J + j] = make_float2((float)std::cos(th), (float)std::sin(th));
      }
    }
    // pageable source: the copy is staged before the call returns
    e = cudaMemcpyAsync(ws + L.rope[a], tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) {
      delete r;
      return cuda_fail(e);
    }
  }
  if (!encode_maps(r)) {
    delete r;
    return cuda_fail(cudaErrorInvalidValue);
  }
  if ((e = prepare_attend(rv.D)) != cudaSuccess) {
    delete r;
    return cuda_fail(e);
  }
  *out = r;
  return KVRING_OK;
}

int kvring_write(kvring* r, const void* k, const void* v, const int32_t* pos, int32_t n_new,
                 kvring_stream stream) {
  if (!r || !k || !v || !pos) return KVRING_ERR_INVALID_ARG;
  if (n_new < 1 || n_new > r->rv.S - r->rv.G) return KVRING_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(pos, 4)) return KVRING_ERR_MISALIGNED;
  if (r->rv.G > 0 && !r->globals_written) return KVRING_ERR_SEQUENCE;
  const cudaError_t e =
      launch_ring_kv_write(r->rv, k, v, pos, n_new, false, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  r->window_written = true;
  return KVRING_OK;
}

int kvring_write_global(kvring* r, const void* k, const void* v, const int32_t* pos, int32_t n,
                        kvring_stream stream) {
  if (!r || !k || !v || !pos) return KVRING_ERR_INVALID_ARG;
  if (r->rv.G == 0 || n != r->rv.G) return KVRING_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(pos, 4)) return KVRING_ERR_MISALIGNED;
  if (r->globals_written || r->window_written) return KVRING_ERR_SEQUENCE;
  const cudaError_t e = launch_ring_kv_write(r->rv, k, v, pos, n, true, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  r->globals_written = true;
  return KVRING_OK;
}

int kvring_reset_positions(kvring* r, int32_t d, kvring_stream stream) {
  if (!r) return KVRING_ERR_INVALID_ARG;
  if (r->cfg.scale_mode == KVRING_SCALES_STATIC && !r->calibrated) return KVRING_ERR_SEQUENCE;
  const cudaError_t e = launch_delta_rerotate(r->rv, delta_table(r->cfg, d), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVRING_OK : cuda_fail(e);
}

int kvring_reset_positions_batch(kvring* const* rings, int32_t n, int32_t d, kvring_stream stream) {
  if (!rings || n < 1) return KVRING_ERR_INVALID_ARG;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const kvring* r0 = rings[0];
  if (!r0) return KVRING_ERR_INVALID_ARG;
  std::vector<const RingView*> rvs((size_t)n);
  for (int i = 0; i < n; ++i) {
    const kvring* r = rings[i];
    if (!r || r->device != dev) return KVRING_ERR_INVALID_ARG;
    // one rotation table for all: the same head_dim, temporal axis and base
    if (r->cfg.head_dim != r0->cfg.head_dim || r->cfg.axis_dims[0] != r0->cfg.axis_dims[0] ||
        r->cfg.rope_base != r0->cfg.rope_base)
      return KVRING_ERR_INVALID_ARG;
    if (r->cfg.scale_mode == KVRING_SCALES_STATIC && !r->calibrated) return KVRING_ERR_SEQUENCE;
    rvs[(size_t)i] = &r->rv;
  }
  e = launch_delta_rerotate_batch(rvs.data(), n, delta_table(r0->cfg, d), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVRING_OK : cuda_fail(e);
}

int kvring_set_qk_norm(kvring* r, const void* gamma_q, const void* gamma_k, float eps) {
  if (!r) return KVRING_ERR_INVALID_ARG;
  if ((gamma_q || gamma_k) && (!(eps > 0.0f) || !std::isfinite(eps))) return KVRING_ERR_INVALID_ARG;
  if (!aligned(gamma_q, 16) || !aligned(gamma_k, 16)) return KVRING_ERR_MISALIGNED;
  // a calibrated ring's fixed K scales were taken from the keys as they were
  // normalised then: the K norm may no longer change
  const bool k_changes = gamma_k != static_cast<const void*>(r->rv.gamma_k) || (gamma_k && eps != r->rv.norm_eps);
  if (r->calibrated && k_changes) return KVRING_ERR_SEQUENCE;
  r->rv.gamma_q = static_cast<const uint4*>(gamma_q);
  r->rv.gamma_k = static_cast<const uint4*>(gamma_k);
  r->rv.norm_eps = eps;
  return KVRING_OK;
}

int kvring_calibrate(kvring* r, float margin, kvring_stream stream) {
  if (!r) return KVRING_ERR_INVALID_ARG;
  if (!(margin > 0.0f) || !std::isfinite(margin)) return KVRING_ERR_INVALID_ARG;
  if (r->cfg.scale_mode != KVRING_SCALES_STATIC || r->calibrated || !(r->globals_written || r->window_written))
    return KVRING_ERR_SEQUENCE;
  const cudaError_t e = launch_calibrate(r->rv, margin, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  r->calibrated = true;
  return KVRING_OK;
}

int kvring_attend(kvring* r, const void* q, const int32_t* q_pos, int32_t n_q, void* out, kvring_stream stream) {
  if (!r || !q || !q_pos || !out) return KVRING_ERR_INVALID_ARG;
  if (n_q < 1 || n_q > r->cfg.max_queries) return KVRING_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(q_pos, 4)) return KVRING_ERR_MISALIGNED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_q_prep(r->rv, q, q_pos, n_q, st);
  if (e == cudaSuccess)
    e = launch_fp8_ring_attn(r->rv, r->maps, r->q_map, n_q, out, r->cfg.out_dtype == KVRING_OUT_F32, st);
  return e == cudaSuccess ? KVRING_OK : cuda_fail(e);
}

int kvring_attend_noalloc(kvring* r, const void* q, const int32_t* q_pos, int32_t n_q, void* out,
                          kvring_stream stream) {
  if (!r || !q || !q_pos || !out) return KVRING_ERR_INVALID_ARG;
  if (n_q < 1) return KVRING_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(q_pos, 4)) return KVRING_ERR_MISALIGNED;
  // scratch layout: e4m3 codes [n_q][H][D], then fp32 scales [H][round_up(n_q, 4)],
  // then the per-head attention range factors fp32 [H][2]
  const size_t H = r->rv.H, D = r->rv.D;
  const size_t q_pad = round_up((size_t)n_q, 4);
  const size_t scale_off = round_up((size_t)n_q * H * D, 1024);
  const size_t stat_off = scale_off + H * q_pad * sizeof(float);
  if (stat_off + 2 * H * sizeof(float) > (size_t)KVRING_NOALLOC_SCRATCH_BYTES) return KVRING_ERR_SCRATCH_LIMIT;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev != r->device) return KVRING_ERR_INVALID_ARG;
  uint8_t* scratch = nullptr;
  const int s = noalloc_scratch(dev, &scratch);
  if (s != KVRING_OK) return s;
  RingView rv = r->rv;
  rv.q_codes = scratch;
  rv.q_scale = reinterpret_cast<float*>(scratch + scale_off);
  rv.head_stat = reinterpret_cast<float*>(scratch + stat_off);
  rv.Q_pad = (int)q_pad;
  CUtensorMap q_map;
  if (!encode_query_map(&q_map, scratch, rv.H, rv.D, n_q)) return cuda_fail(cudaErrorInvalidValue);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  e = launch_q_prep(rv, q, q_pos, n_q, st);
  if (e == cudaSuccess)
    e = launch_fp8_ring_attn(rv, r->maps, q_map, n_q, out, r->cfg.out_dtype == KVRING_OUT_F32, st);
  return e == cudaSuccess ? KVRING_OK : cuda_fail(e);
}

int kvring_destroy(kvring* r) {
  delete r;
  return KVRING_OK;
}

const char* kvring_status_string(int s) {
  switch (s) {
    case KVRING_OK: return "ok";
    case KVRING_ERR_INVALID_ARG: return "invalid argument";
    case KVRING_ERR_MISALIGNED: return "misaligned pointer";
    case KVRING_ERR_UNSUPPORTED: return "unsupported shape";
    case KVRING_ERR_CUDA: return "CUDA error";
    case KVRING_ERR_WORKSPACE: return "workspace too small";
    case KVRING_ERR_NO_DEVICE: return "no sm_100-family device is current";
    case KVRING_ERR_SCRATCH_LIMIT:
      return "request larger than the static scratch of kvring_attend_noalloc (KVRING_NOALLOC_SCRATCH_BYTES)";
    case KVRING_ERR_SEQUENCE:
      return "call out of order (global slots: once, before the first window write; fixed scales: "
             "calibrate once, after a write and before the first reset)";
    default: return "unknown status";
  }
}

int kvring_last_cuda_error(void) { return g_last_cuda_error; }

int kvring_layout(const kvring* r, void** k_codes, void** v_codes, void** k_scales, void** v_scales, void** state,
                  int32_t* s_pad) {
  if (!r) return KVRING_ERR_INVALID_ARG;
  if (k_codes) *k_codes = r->rv.k_codes;
  if (v_codes) *v_codes = r->rv.v_codes;
  if (k_scales) *k_scales = r->rv.k_scale;
  if (v_scales) *v_scales = r->rv.v_scale;
  if (state) *state = r->rv.state;
  if (s_pad) *s_pad = r->rv.S_pad;
  return KVRING_OK;
}

int kvring_debug_state(const kvring* r, kvring_stream stream, int32_t* out3) {
  if (!r || !out3) return KVRING_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int32_t w[3];
  e = cudaMemcpy(w, r->rv.state, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  out3[0] = w[ST_WP];
  out3[1] = w[ST_NVALID];
  out3[2] = w[ST_ERR];
  return KVRING_OK;
}

int kvring_debug_wait_timeout(int64_t limit_ns, int32_t complete, int64_t* out2, kvring_stream stream) {
  if (!out2 || limit_ns < 1 || limit_ns > 10000000000ll) return KVRING_ERR_INVALID_ARG;
  if (!aligned(out2, 8)) return KVRING_ERR_MISALIGNED;
  const cudaError_t e = launch_debug_wait(limit_ns, complete != 0, out2, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVRING_OK : cuda_fail(e);
}

int kvring_debug_quantize(const float* x, int64_t rows, int32_t d, uint8_t* codes, float* scales,
                          kvring_stream stream) {
  if (!x || !codes || !scales || rows < 1) return KVRING_ERR_INVALID_ARG;
  if (d != 16 && d != 32 && d != 64 && d != 128 && d != 256) return KVRING_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return KVRING_ERR_MISALIGNED;
  const cudaError_t e = launch_debug_quantize(x, rows, d, codes, scales, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVRING_OK : cuda_fail(e);
}

}  // extern "C"
