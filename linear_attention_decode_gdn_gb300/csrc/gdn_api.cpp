// gdn_api.cpp -- the extern "C" entry points declared in include/gdn.h:
// argument validation, kernel selection and error reporting. No allocation.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <cuda_runtime_api.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

thread_local char g_last_error[512] = "";

constexpr uint32_t kKnownFlags = GDN_QKV_BF16 | GDN_FUSE_CONV | GDN_NO_QK_L2NORM | GDN_GATE_RAW |
                                 GDN_PLAIN_UPDATE | GDN_KLOG_FP32 | GDN_KLOG_PRENORM | GDN_ULOG_BF16 |
                                 GDN_GATE_KDA | GDN_OUT_NORM_GATE | GDN_SPLIT_DV |
                                 GDN_TEST_STARVE_WAIT;
constexpr int kMaxLogCapacity = 63;

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

constexpr int kMaxVerifyTokens = 16;  // positions per request in one verify call

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }

// What a call needs of dk and dv: the decode steps run every shape with a kernel
// (gdn::decode_shape_built: square heads of 16..128, dk = 128 / dv = 64, dk = 64 / dv = 128,
// and square heads of 64 or 128 split along dv); the host-side log sizes and the slot reset
// accept the same shapes; the input stage, verify and prefill square heads only.
enum class Shapes { kDecode, kSquare };

int check_dims(const gdn_dims* d, bool log_call, Shapes shapes = Shapes::kSquare) {
  if (d == nullptr) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
  if (d->batch < 0 || d->num_heads <= 0 || d->dk <= 0 || d->dv <= 0 || d->num_slots <= 0)
    return fail(GDN_ERR_INVALID_ARG, "batch must be >= 0 and num_heads, dk, dv, num_slots > 0");
  if (d->decay_per_key != 0 && d->decay_per_key != 1)
    return fail(GDN_ERR_INVALID_ARG, "decay_per_key must be 0 or 1");
  if ((d->flags & ~kKnownFlags) != 0u) return fail(GDN_ERR_INVALID_ARG, "unknown flag bits");
  const int ns = (d->flags & GDN_SPLIT_DV) ? 2 : 1;
  if (shapes == Shapes::kDecode) {
    if (!gdn::decode_shape_built(d->dk, d->dv, ns))
      return fail(GDN_ERR_UNSUPPORTED,
                  "decode shape dk=%d dv=%d%s not built (dk == dv in {16,32,64,128}, dk=128/dv=64, "
                  "dk=64/dv=128; GDN_SPLIT_DV: dk == dv in {64,128})",
                  d->dk, d->dv, ns > 1 ? " split along dv" : "");
    if (ns > 1 && (d->flags & (GDN_GATE_KDA | GDN_OUT_NORM_GATE)))
      return fail(GDN_ERR_UNSUPPORTED, "GDN_SPLIT_DV is built without the KDA gate and output epilogue");
  } else {
    if (d->dk != d->dv || (d->dk != 16 && d->dk != 32 && d->dk != 64 && d->dk != 128))
      return fail(GDN_ERR_UNSUPPORTED, "head size dk=%d dv=%d not built for this call (dk == dv in {16,32,64,128})",
                  d->dk, d->dv);
    if (ns > 1) return fail(GDN_ERR_UNSUPPORTED, "GDN_SPLIT_DV applies to the decode steps only");
  }
  if (static_cast<long long>(d->batch) * d->num_heads > 0x3fffffffLL)
    return fail(GDN_ERR_INVALID_ARG, "batch * num_heads too large");
  if (log_call) {
    if (d->log_capacity < 0) return fail(GDN_ERR_INVALID_ARG, "log_capacity < 0");
    if (d->log_capacity > kMaxLogCapacity)
      return fail(GDN_ERR_UNSUPPORTED, "log_capacity %d > %d", d->log_capacity, kMaxLogCapacity);
  }
  if ((d->flags & GDN_KLOG_PRENORM) &&
      ((d->flags & GDN_FUSE_CONV) || (d->flags & GDN_NO_QK_L2NORM)))
    return fail(GDN_ERR_UNSUPPORTED, "GDN_KLOG_PRENORM needs L2 normalisation and no fused conv");
  if ((d->flags & GDN_GATE_KDA) && (d->flags & GDN_GATE_RAW))
    return fail(GDN_ERR_INVALID_ARG, "GDN_GATE_KDA and GDN_GATE_RAW exclude each other");
  return GDN_OK;
}

int check_gate_inputs(const gdn_dims* d, const gdn_inputs* in) {
  if ((d->flags & GDN_GATE_KDA) && (in->a_log == nullptr || in->dt_bias == nullptr))
    return fail(GDN_ERR_INVALID_ARG, "GDN_GATE_KDA needs a_log and dt_bias");
  if ((d->flags & GDN_OUT_NORM_GATE) && in->out_gate == nullptr)
    return fail(GDN_ERR_INVALID_ARG, "GDN_OUT_NORM_GATE needs out_gate");
  return GDN_OK;
}

int check_inputs(const gdn_dims* d, const gdn_inputs* in) {
  if (in == nullptr) return fail(GDN_ERR_INVALID_ARG, "inputs is NULL");
  if (int rc = check_gate_inputs(d, in)) return rc;
  if (in->slot == nullptr || in->log_decay == nullptr)
    return fail(GDN_ERR_INVALID_ARG, "slot and log_decay are required");
  if (d->flags & GDN_FUSE_CONV) {
    if (in->mixed_qkv == nullptr || in->conv_w == nullptr || in->conv_pool == nullptr)
      return fail(GDN_ERR_INVALID_ARG, "GDN_FUSE_CONV needs mixed_qkv, conv_w and conv_pool");
    if (!aligned16(in->mixed_qkv) || !aligned16(in->conv_w))
      return fail(GDN_ERR_UNSUPPORTED, "mixed_qkv and conv_w must be 16-byte aligned");
  } else {
    if (in->q == nullptr || in->k == nullptr || in->v == nullptr)
      return fail(GDN_ERR_INVALID_ARG, "q, k and v are required");
    if (!aligned16(in->q) || !aligned16(in->k) || !aligned16(in->v))
      return fail(GDN_ERR_UNSUPPORTED, "q, k and v must be 16-byte aligned");
  }
  return GDN_OK;
}

int check_log(const gdn_dims* d, const gdn_log* log) {
  if (log == nullptr) return fail(GDN_ERR_INVALID_ARG, "log is NULL");
  if (log->len == nullptr || log->ell == nullptr)
    return fail(GDN_ERR_INVALID_ARG, "log->len and log->ell are required");
  if (d->log_capacity > 0) {
    if (log->k_log == nullptr || log->u_log == nullptr || log->lam_log == nullptr)
      return fail(GDN_ERR_INVALID_ARG, "k_log, u_log and lam_log are required when log_capacity > 0");
    if (!aligned16(log->k_log) || !aligned16(log->u_log))
      return fail(GDN_ERR_UNSUPPORTED, "k_log and u_log must be 16-byte aligned");
  }
  return GDN_OK;
}

gdn::DecodeParams make_params(const gdn_dims* d, const gdn_inputs* in) {
  gdn::DecodeParams p{};
  p.B = d->batch;
  p.H = d->num_heads;
  p.D = d->dk;
  p.DV = d->dv;
  p.num_slots = d->num_slots;
  p.C = d->log_capacity;
  p.dlam = d->decay_per_key ? d->dk : 1;
  p.channels = 2 * d->num_heads * d->dk + d->num_heads * d->dv;
  p.flags = d->flags;
  p.q_scale = d->q_scale;
  p.l2_eps = d->l2_eps;
  p.q = in->q;
  p.k = in->k;
  p.v = in->v;
  p.mixed = in->mixed_qkv;
  p.conv_w = in->conv_w;
  p.conv_b = in->conv_b;
  p.conv_pool = in->conv_pool;
  p.lam = in->log_decay;
  p.beta = in->beta;
  p.slot = in->slot;
  p.a_log = in->a_log;
  p.dt_bias = in->dt_bias;
  p.out_gate = in->out_gate;
  p.out_norm_w = in->out_norm_w;
  p.lower_bound = d->gate_lower_bound;
  p.out_eps = d->out_eps;
  return p;
}

int launched(cudaError_t err, const char* what) {
  if (err != cudaSuccess)
    return fail(GDN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
  g_last_error[0] = '\0';
  return GDN_OK;
}

int decode_common(int mode, const gdn_dims* dims, const gdn_inputs* in, float* pool,
                  const gdn_log* log, float* o, int32_t* status, void* stream, const char* name) {
  const bool log_call = mode != gdn::MODE_DENSE;
  int rc = check_dims(dims, log_call, Shapes::kDecode);
  if (rc != GDN_OK) return rc;
  if (dims->batch == 0) return GDN_OK;
  if ((rc = check_inputs(dims, in)) != GDN_OK) return rc;
  if (pool == nullptr || o == nullptr) return fail(GDN_ERR_INVALID_ARG, "state/base pool and o are required");
  if (!aligned16(pool) || !aligned16(o))
    return fail(GDN_ERR_UNSUPPORTED, "state/base pool and o must be 16-byte aligned");
  if (log_call && (rc = check_log(dims, log)) != GDN_OK) return rc;
  if (mode == gdn::MODE_APPEND && dims->log_capacity < 1)
    return fail(GDN_ERR_INVALID_ARG, "append needs log_capacity >= 1");
  // the split path addresses the pool's rows with 32-bit tensor-copy coordinates
  if ((dims->flags & GDN_SPLIT_DV) &&
      static_cast<long long>(dims->num_slots) * dims->num_heads * dims->dk > 0x7fffffffLL)
    return fail(GDN_ERR_UNSUPPORTED, "GDN_SPLIT_DV: num_slots * num_heads * dk must stay below 2^31");
  if (gdn::decode_smem_bytes(mode, dims->dk, dims->dv, (dims->flags & GDN_SPLIT_DV) ? 2 : 1,
                             log_call ? dims->log_capacity : 0,
                             dims->decay_per_key ? dims->dk : 1,
                             (dims->flags & GDN_KLOG_FP32) ? 4 : 2,
                             (dims->flags & GDN_ULOG_BF16) ? 2 : 4) == 0)
    return fail(GDN_ERR_UNSUPPORTED, "log_capacity %d does not fit in shared memory for this shape",
                dims->log_capacity);
  gdn::DecodeParams p = make_params(dims, in);
  p.state = pool;
  p.o = o;
  p.status = status;
  if (log_call) {
    p.k_log = log->k_log;
    p.u_log = log->u_log;
    p.lam_log = log->lam_log;
    p.ell = log->ell;
    p.len = log->len;
  }
  return launched(gdn::launch_decode(mode, p, static_cast<cudaStream_t>(stream)), name);
}

}  // namespace

extern "C" {

int gdn_version(void) { return GDN_API_VERSION; }

const char* gdn_strerror(int code) {
  switch (code) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported shape, flag combination or alignment";
    case GDN_ERR_CUDA: return "CUDA launch failure";
    default: return "unknown error code";
  }
}

const char* gdn_last_error(void) { return g_last_error; }

int gdn_conv_l2norm(const gdn_dims* dims, const gdn_inputs* in, float* q_out, float* k_out,
                    float* v_out, int32_t* status, void* stream) {
  int rc = check_dims(dims, false);
  if (rc != GDN_OK) return rc;
  if (!(dims->flags & GDN_FUSE_CONV))
    return fail(GDN_ERR_INVALID_ARG, "gdn_conv_l2norm needs GDN_FUSE_CONV in dims->flags");
  if (dims->batch == 0) return GDN_OK;
  if ((rc = check_inputs(dims, in)) != GDN_OK) return rc;
  if (q_out == nullptr || k_out == nullptr || v_out == nullptr)
    return fail(GDN_ERR_INVALID_ARG, "q_out, k_out and v_out are required");
  gdn::DecodeParams p = make_params(dims, in);
  p.q_out = q_out;
  p.k_out = k_out;
  p.v_out = v_out;
  p.status = status;
  return launched(gdn::launch_conv_l2norm(p, static_cast<cudaStream_t>(stream)), "gdn_conv_l2norm");
}

int gdn_decode_dense(const gdn_dims* dims, const gdn_inputs* in, float* state_pool, float* o,
                     int32_t* status, void* stream) {
  return decode_common(gdn::MODE_DENSE, dims, in, state_pool, nullptr, o, status, stream,
                       "gdn_decode_dense");
}

int gdn_decode_append(const gdn_dims* dims, const gdn_inputs* in, const float* base_pool,
                      const gdn_log* log, float* o, int32_t* status, void* stream) {
  // The append kernel only reads the base.
  return decode_common(gdn::MODE_APPEND, dims, in, const_cast<float*>(base_pool), log, o, status,
                       stream, "gdn_decode_append");
}

int gdn_decode_merge(const gdn_dims* dims, const gdn_inputs* in, float* base_pool,
                     const gdn_log* log, float* o, int32_t* status, void* stream) {
  return decode_common(gdn::MODE_MERGE, dims, in, base_pool, log, o, status, stream,
                       "gdn_decode_merge");
}

int gdn_decode_step(const gdn_dims* dims, const gdn_inputs* in, float* base_pool,
                    const gdn_log* log, float* o, int32_t* status, void* stream) {
  return decode_common(gdn::MODE_STEP, dims, in, base_pool, log, o, status, stream,
                       "gdn_decode_step");
}

int gdn_decode_verify(const gdn_dims* dims, int32_t num_tokens, const gdn_inputs* in,
                      const int32_t* state_indices, const int32_t* num_accepted, float* state_pool,
                      float* o, int32_t* status, void* stream) {
  int rc = check_dims(dims, false);
  if (rc != GDN_OK) return rc;
  if (num_tokens < 1 || num_tokens > kMaxVerifyTokens)
    return fail(GDN_ERR_UNSUPPORTED, "num_tokens %d outside [1, %d]", num_tokens, kMaxVerifyTokens);
  if (dims->flags & (GDN_KLOG_FP32 | GDN_KLOG_PRENORM | GDN_ULOG_BF16 | GDN_TEST_STARVE_WAIT))
    return fail(GDN_ERR_UNSUPPORTED, "verify runs the dense recurrence: no log flags");
  if (static_cast<long long>(dims->batch) * num_tokens * dims->num_heads > 0x7fffffffLL)
    return fail(GDN_ERR_INVALID_ARG, "batch * num_tokens * num_heads too large");
  if (dims->batch == 0) return GDN_OK;
  if (in == nullptr || in->log_decay == nullptr)
    return fail(GDN_ERR_INVALID_ARG, "inputs and log_decay are required");
  if ((rc = check_gate_inputs(dims, in)) != GDN_OK) return rc;
  if (dims->flags & GDN_FUSE_CONV) {
    if (in->mixed_qkv == nullptr || in->conv_w == nullptr || in->conv_pool == nullptr)
      return fail(GDN_ERR_INVALID_ARG, "GDN_FUSE_CONV needs mixed_qkv, conv_w and conv_pool");
    if (!aligned16(in->mixed_qkv) || !aligned16(in->conv_w))
      return fail(GDN_ERR_UNSUPPORTED, "mixed_qkv and conv_w must be 16-byte aligned");
  } else {
    if (in->q == nullptr || in->k == nullptr || in->v == nullptr)
      return fail(GDN_ERR_INVALID_ARG, "q, k and v are required");
    if (!aligned16(in->q) || !aligned16(in->k) || !aligned16(in->v))
      return fail(GDN_ERR_UNSUPPORTED, "q, k and v must be 16-byte aligned");
  }
  if (state_indices == nullptr || num_accepted == nullptr || state_pool == nullptr || o == nullptr)
    return fail(GDN_ERR_INVALID_ARG, "state_indices, num_accepted, state_pool and o are required");
  if (!aligned16(state_pool) || !aligned16(o))
    return fail(GDN_ERR_UNSUPPORTED, "state_pool and o must be 16-byte aligned");
  gdn::DecodeParams p = make_params(dims, in);
  p.T = num_tokens;
  p.state_indices = state_indices;
  p.num_accepted = num_accepted;
  p.state = state_pool;
  p.o = o;
  p.status = status;
  return launched(gdn::launch_verify(p, static_cast<cudaStream_t>(stream)), "gdn_decode_verify");
}

int gdn_prefill(const gdn_dims* dims, int32_t num_tokens, const gdn_inputs* in, const int32_t* seq_lens,
                float* state_pool, float* o, int32_t* status, void* stream) {
  int rc = check_dims(dims, false);
  if (rc != GDN_OK) return rc;
  if (num_tokens < 0) return fail(GDN_ERR_INVALID_ARG, "num_tokens < 0");
  if (dims->flags & (GDN_KLOG_FP32 | GDN_KLOG_PRENORM | GDN_ULOG_BF16 | GDN_TEST_STARVE_WAIT))
    return fail(GDN_ERR_UNSUPPORTED, "prefill: no DeltaLog flags");
  if (static_cast<long long>(dims->batch) * num_tokens * dims->num_heads > 0x7fffffffLL)
    return fail(GDN_ERR_INVALID_ARG, "batch * num_tokens * num_heads too large");
  if (dims->batch == 0 || num_tokens == 0) return GDN_OK;
  if ((rc = check_inputs(dims, in)) != GDN_OK) return rc;
  if (state_pool == nullptr || o == nullptr) return fail(GDN_ERR_INVALID_ARG, "state_pool and o are required");
  if (!aligned16(state_pool)) return fail(GDN_ERR_UNSUPPORTED, "state_pool must be 16-byte aligned");
  gdn::DecodeParams p = make_params(dims, in);
  p.T = num_tokens;
  p.seq_lens = seq_lens;
  p.state = state_pool;
  p.o = o;
  p.status = status;
  return launched(gdn::launch_prefill(p, static_cast<cudaStream_t>(stream)), "gdn_prefill");
}

int gdn_log_bytes(const gdn_dims* dims, gdn_log_sizes* out) {
  int rc = check_dims(dims, true, Shapes::kDecode);
  if (rc != GDN_OK) return rc;
  if (out == nullptr) return fail(GDN_ERR_INVALID_ARG, "out is NULL");
  const size_t sh = static_cast<size_t>(dims->num_slots) * dims->num_heads;
  const size_t C = static_cast<size_t>(dims->log_capacity);
  const size_t dlam = dims->decay_per_key ? static_cast<size_t>(dims->dk) : 1u;
  const size_t kb = (dims->flags & GDN_KLOG_FP32) ? 4u : 2u;
  out->k_log = sh * C * dims->dk * kb;
  out->u_log = sh * C * dims->dv * ((dims->flags & GDN_ULOG_BF16) ? 2u : 4u);
  out->lam_log = sh * C * dlam * 4u;
  out->ell = sh * dlam * 4u;
  out->len = sh * 4u;
  out->residency = out->k_log + out->u_log + out->lam_log + out->ell;
  out->total = out->residency + out->len;
  return GDN_OK;
}

int gdn_slot_reset(const gdn_dims* dims, const gdn_log* log, void* conv_pool, float* state_pool,
                   const int32_t* slots, int32_t n, int32_t* status, void* stream) {
  int rc = check_dims(dims, false, Shapes::kDecode);
  if (rc != GDN_OK) return rc;
  if (n < 0) return fail(GDN_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return GDN_OK;
  if (slots == nullptr) return fail(GDN_ERR_INVALID_ARG, "slots is NULL");
  if (state_pool != nullptr && !aligned16(state_pool))
    return fail(GDN_ERR_UNSUPPORTED, "state_pool must be 16-byte aligned");
  gdn::ResetParams p{};
  p.H = dims->num_heads;
  p.D = dims->dk;
  p.DV = dims->dv;
  p.num_slots = dims->num_slots;
  p.dlam = dims->decay_per_key ? dims->dk : 1;
  p.channels = 2 * dims->num_heads * dims->dk + dims->num_heads * dims->dv;
  p.n = n;
  p.flags = dims->flags;
  p.slots = slots;
  p.ell = log ? log->ell : nullptr;
  p.len = log ? log->len : nullptr;
  p.conv_pool = conv_pool;
  p.state = state_pool;
  p.status = status;
  return launched(gdn::launch_slot_reset(p, static_cast<cudaStream_t>(stream)), "gdn_slot_reset");
}

}  // extern "C"
