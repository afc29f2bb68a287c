// gdn_conv.cu -- the input stage as its own kernel (gdn_conv_l2norm) and the
// slot-reset kernel (gdn_slot_reset).
#include "gdn_device.cuh"

namespace gdn {

// One CTA per (request, head): width-4 conv + SiLU of the head's q, k, v
// channels, conv cache shift, then q, k L2-normalised (appendix 附2 of the
// evolution article) and q scaled. Same thread roles as the decode kernel.
__global__ void __launch_bounds__(NT) gdn_conv_l2norm_kernel(const DecodeParams p) {
  __shared__ float part[NW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / p.H;
  const int h = blockIdx.x - b * p.H;
  const int slot = __ldg(p.slot + b);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (tid == 0) atomic_status(p.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  const int D = p.D;
  float x, vj;
  load_token(p, b, h, slot, tid, &x, &vj);
  const float ss = warp_sum(x * x);
  if (lane == 0) part[warp] = ss;
  __syncthreads();
  conv_commit(p, b, h, slot, tid);
  const bool l2 = (p.flags & GDN_NO_QK_L2NORM) == 0u;
  const float qinv = l2 ? 1.0f / sqrtf(part[0] + part[1] + part[2] + part[3] + p.l2_eps) : 1.0f;
  const float kinv = l2 ? 1.0f / sqrtf(part[4] + part[5] + part[6] + part[7] + p.l2_eps) : 1.0f;
  const size_t row = (static_cast<size_t>(b) * p.H + h) * D;
  if (tid < D) {
    p.q_out[row + tid] = x * qinv * p.q_scale;
    p.v_out[row + tid] = vj;
  } else if (tid >= 128 && tid < 128 + D) {
    p.k_out[row + tid - 128] = x * kinv;
  }
}

// grid (n, parts): block (i, part) clears its share of slot slots[i].
__global__ void __launch_bounds__(NT) gdn_slot_reset_kernel(const ResetParams p) {
  const int slot = __ldg(p.slots + blockIdx.x);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (blockIdx.y == 0 && threadIdx.x == 0) atomic_status(p.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  const int tid = threadIdx.x;
  const int part = blockIdx.y, parts = gridDim.y;
  if (part == 0) {
    if (p.len != nullptr)
      for (int i = tid; i < p.H; i += NT) p.len[static_cast<size_t>(slot) * p.H + i] = 0;
    if (p.ell != nullptr)
      for (int i = tid; i < p.H * p.dlam; i += NT)
        p.ell[static_cast<size_t>(slot) * p.H * p.dlam + i] = 0.0f;
  }
  if (p.conv_pool != nullptr) {
    const size_t n = static_cast<size_t>(p.channels) * 3;
    const size_t per = (n + parts - 1) / parts;
    const size_t lo = per * part, hi = lo + per < n ? lo + per : n;
    if (p.flags & GDN_QKV_BF16) {
      uint16_t* row = static_cast<uint16_t*>(p.conv_pool) + static_cast<size_t>(slot) * n;
      for (size_t i = lo + tid; i < hi; i += NT) row[i] = 0;
    } else {
      float* row = static_cast<float*>(p.conv_pool) + static_cast<size_t>(slot) * n;
      for (size_t i = lo + tid; i < hi; i += NT) row[i] = 0.0f;
    }
  }
  if (p.state != nullptr) {
    const size_t n4 = static_cast<size_t>(p.H) * p.D * p.DV / 4;
    float4* row = reinterpret_cast<float4*>(p.state) + static_cast<size_t>(slot) * n4;
    const size_t per = (n4 + parts - 1) / parts;
    const size_t lo = per * part, hi = lo + per < n4 ? lo + per : n4;
    for (size_t i = lo + tid; i < hi; i += NT) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

cudaError_t launch_conv_l2norm(const DecodeParams& p, cudaStream_t stream) {
  gdn_conv_l2norm_kernel<<<dim3(static_cast<unsigned>(p.B * p.H)), dim3(NT), 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_slot_reset(const ResetParams& p, cudaStream_t stream) {
  gdn_slot_reset_kernel<<<dim3(static_cast<unsigned>(p.n), 16u), dim3(NT), 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
