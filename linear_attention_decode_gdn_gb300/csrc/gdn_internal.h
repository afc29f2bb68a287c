// gdn_internal.h -- launch parameters shared by the C-ABI layer and the kernels.
// Not part of the public interface (include/gdn.h is).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime_api.h>

namespace gdn {

// Which path of Algorithm 1 (DeltaLog notes, Sec. 2.3) a launch takes.
enum Mode : int {
  MODE_DENSE = 0,   // full state read + write every token
  MODE_APPEND = 1,  // base read only, one log entry written
  MODE_MERGE = 2,   // base read, log + current token folded into the base (Eq. (6))
  MODE_STEP = 3,    // per slot-head: append if L < C on entry, else merge
};

struct DecodeParams {
  int32_t B, H, D, num_slots, C, dlam, channels;
  int32_t DV;              // value head size (D is the key head size)
  int32_t prefetch_ahead;  // decode: CTAs resident at once (one wave); CTA i prefetches the inputs
                           // of item i + this into L2, the first wave its own tile (0: off)
  uint32_t flags;
  float q_scale, l2_eps;
  const void* q;
  const void* k;
  const void* v;
  const void* mixed;
  const float* conv_w;
  const float* conv_b;
  void* conv_pool;
  const float* lam;
  const float* beta;
  const int32_t* slot;
  float* state;  // dense: state pool; DeltaLog: base pool
  void* k_log;
  void* u_log;
  float* lam_log;
  float* ell;
  int32_t* len;
  float* o;
  int32_t* status;
  // KDA gate parametrisation and output epilogue
  const float* a_log;
  const float* dt_bias;
  const float* out_gate;
  const float* out_norm_w;
  float lower_bound, out_eps;
  // verify: positions per request, [B][T] pool rows, [B] accepted counts
  int32_t T;
  const int32_t* state_indices;
  const int32_t* num_accepted;
  // prefill: [B] prompt lengths (NULL: all T)
  const int32_t* seq_lens;
  // conv_l2norm outputs
  float* q_out;
  float* k_out;
  float* v_out;
};

struct ResetParams {
  int32_t H, D, DV, num_slots, dlam, channels, n;
  uint32_t flags;
  const int32_t* slots;
  float* ell;
  int32_t* len;
  void* conv_pool;
  float* state;
  int32_t* status;
};

// Kernel launchers (defined in the .cu files). Return cudaSuccess or the launch error.
cudaError_t launch_decode(int mode, const DecodeParams& p, cudaStream_t stream);
// the shapes gdn_decode.cu does not instantiate (dk != dv; heads split along dv)
cudaError_t launch_decode_x(int mode, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_conv_l2norm(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_slot_reset(const ResetParams& p, cudaStream_t stream);
cudaError_t launch_verify(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_prefill(const DecodeParams& p, cudaStream_t stream);
// the tensor-core prefill (head size 128, per-head decay, no fused conv / KDA gate / epilogue)
bool prefill_tc_supported(const DecodeParams& p);
cudaError_t launch_prefill_tc(const DecodeParams& p, cudaStream_t stream);
bool prefill_tc_pk_supported(const DecodeParams& p);
cudaError_t launch_prefill_tc_pk(const DecodeParams& p, cudaStream_t stream);

// Dynamic shared memory of a prefill CTA (bytes).
size_t prefill_smem_bytes(int D, int dlam);

// the dynamic shared memory of those shapes (bytes)
size_t decode_smem_bytes_x(int mode, int dk, int dv, int ns, int C, int klog_bytes, int ulog_bytes);

// Decode shapes with kernels: dk x dv heads, ns CTAs per head along dv.
bool decode_shape_built(int dk, int dv, int ns);
// Dynamic shared memory a decode launch needs (bytes); 0 if the shape is not built.
size_t decode_smem_bytes(int mode, int dk, int dv, int ns, int C, int dlam, int klog_bytes, int ulog_bytes);

}  // namespace gdn
