// Host-side entry points of the kernels (internal to libkvring).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace kvring_dev {

// cos/sin of the reset rotation -d * omega_{0,j} for the temporal pairs j,
// formed in fp64 on the host and rounded once to fp32.
struct DeltaTable {
  float2 cs[64];
  int n_pairs;
};

// What the rotation of one ring's keys needs (a slice of RingView).
struct RotRing {
  uint8_t* k_codes;
  float* k_scale;
  int32_t* state;
  const float* stat;
  int32_t H, S, S_pad, G, scale_mode;
};

// Rings rotated by one launch (kernel parameters).
constexpr int kMaxBatchRings = 32;
struct RotBatch {
  RotRing r[kMaxBatchRings];
};

// Slots per key tile of the attention kernel (the box height of its K, V and
// scale tensor maps).
constexpr int kAttnKeyTile = 128;

struct AttnMaps {
  CUtensorMap k_codes;   // [H][S][D] u8, box {D, kAttnKeyTile, 1}
  CUtensorMap v_codes;
  CUtensorMap k_scale;   // [H][S_pad] f32, box {kAttnKeyTile, 1}
  CUtensorMap v_scale;
};

// Launch with programmatic stream serialisation (the kernel calls pdl_wait
// before touching global memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// glob: the G global tokens into slots 0 .. G-1 (else a window write)
cudaError_t launch_ring_kv_write(const RingView& rv, const void* k, const void* v, const int32_t* pos, int n_new,
                                 bool glob, cudaStream_t st);
cudaError_t launch_delta_rerotate(const RingView& rv, const DeltaTable& dt, cudaStream_t st);
// the same rotation over n rings of one head_dim, kMaxBatchRings per launch
cudaError_t launch_delta_rerotate_batch(const RingView* const* rvs, int n, const DeltaTable& dt, cudaStream_t st);
// per-head fixed scales from the recorded maxima, then every valid row re-quantised with them
cudaError_t launch_calibrate(const RingView& rv, float margin, cudaStream_t st);
// one block whose warps wait on a barrier (complete: it is also completed);
// out2 = {error bits, nanoseconds waited}
cudaError_t launch_debug_wait(long long limit_ns, bool complete, int64_t* out2, cudaStream_t st);
cudaError_t launch_debug_quantize(const float* x, long long rows, int d, uint8_t* codes, float* scales,
                                  cudaStream_t st);
cudaError_t launch_q_prep(const RingView& rv, const void* q, const int32_t* q_pos, int n_q, cudaStream_t st);
cudaError_t prepare_attend(int D);   // once per device: opt in to the kernel's shared memory
// tmQ: the query codes of this call (rv.q_codes), [n_q][H][D] u8, box {D, 1, 128}
cudaError_t launch_fp8_ring_attn(const RingView& rv, const AttnMaps& maps, const CUtensorMap& tmQ, int n_q, void* out,
                                 int out_f32, cudaStream_t st);

}  // namespace kvring_dev
