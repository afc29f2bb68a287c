// gdn_verify.cu -- speculative-decoding verification on the dense state.
//
// Inference handbook, "推测解码：验证后如何恢复状态": a verify step feeds T positions
// per request (the last sampled token and the drafts) through the recurrence and
// keeps the state after every position in its own pool row; the next round starts
// from the row the acceptance count selects, so a rejected draft is rolled back by
// indexing.  Here one CTA owns one (request, head): the initial tile comes in by TMA
// once, the T dense steps run on it in shared memory, and every post-position state
// is stored to its row with 16-byte coalesced stores.  Per position the arithmetic is
// the dense decode step's (decayed-state residual, outer-product write, post-update
// readout; evolution article, "GDN" / "KDA实现逻辑概述").
#include <atomic>

#include "gdn_device.cuh"

namespace gdn {

constexpr int kMaxVerifyTokens = 16;

namespace {

// Widened conv window of one channel (inference handbook, "推测解码：验证后如何恢复状态":
// the conv cache of a verify path holds conv_kernel - 1 + num_spec pre-conv inputs, the
// round's inputs are appended at its end, and the next round starts reading at offset
// num_accepted - 1).  With T positions the window row has T + 2 elements (dtype of the
// inputs), column 0 oldest.  s[0..2] are the three inputs before the current position.
__device__ __forceinline__ float conv_window_load(const void* pool, size_t i, bool bf16) {
  return bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(pool)[i]) : static_cast<const float*>(pool)[i];
}

__device__ __forceinline__ void conv_window_store(void* pool, size_t i, float x, bool bf16) {
  // values that came in as bf16 convert back exactly
  if (bf16)
    static_cast<uint16_t*>(pool)[i] = static_cast<uint16_t>(__float_as_uint(x) >> 16);
  else
    static_cast<float*>(pool)[i] = x;
}

// SiLU(s0 w0 + s1 w1 + s2 w2 + x w3 (+ bias)) of channel c, then the window slides by x
// (same product order as the one-step conv of the decode kernels)
__device__ __forceinline__ float conv_window_step(const DecodeParams& p, int c, float (&s)[3], float x) {
  const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w) + c);
  float acc = s[0] * w.x;
  acc = fmaf(s[1], w.y, acc);
  acc = fmaf(s[2], w.z, acc);
  acc = fmaf(x, w.w, acc);
  if (p.conv_b != nullptr) acc += __ldg(p.conv_b + c);
  s[0] = s[1];
  s[1] = s[2];
  s[2] = x;
  return siluf_(acc);
}

// Shared-memory layout (bytes): tile | mbarriers | scalars | two vector sets | partial sums.
struct VerifyLayout {
  uint32_t tile, bars, scal, vec, red, total;
};

__host__ __device__ inline VerifyLayout verify_layout(int D) {
  VerifyLayout L{};
  uint32_t off = 0;
  L.tile = off;
  off += static_cast<uint32_t>(D * D * 4);
  L.bars = off;
  off += 64;
  L.scal = off;  // int rows[16], int flags, then floats: partials[8], q.k, output-norm partials
  off += 192;
  L.vec = off;   // per position parity: q (later b), k, q*dec, k*dec, dec
  off += static_cast<uint32_t>(2 * 5 * D * 4);
  L.red = off;   // cross-warp partial sums, [4 warps][2][D]
  off += static_cast<uint32_t>(8 * D * 4);
  L.total = off;
  return L;
}

template <int D>
__global__ void __launch_bounds__(NT_DECODE) gdn_verify_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem[];

  constexpr int NCHUNK = (D >= 128) ? 4 : 1;
  constexpr int CHUNK_ROWS = D / NCHUNK;
  constexpr uint32_t CHUNK_BYTES = CHUNK_ROWS * D * 4;
  constexpr int VPR = D / 4;
  constexpr int RPW = 32 / VPR;
  constexpr int RPI = NW * RPW;
  constexpr int NIT = (D + RPI - 1) / RPI;
  constexpr int ITC = NIT / NCHUNK;
  static_assert(NCHUNK == 1 || (NIT % NCHUNK == 0 && CHUNK_ROWS % RPI == 0), "chunking");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool ctrl = warp == NW;
  const int b = blockIdx.x / p.H;
  const int h = blockIdx.x - b * p.H;
  const int T = p.T;
  const int dlam = p.dlam;
  const uint32_t fl = p.flags;

  const VerifyLayout L = verify_layout(D);
  float* tile = reinterpret_cast<float*>(smem + L.tile);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  int* rows_s = reinterpret_cast<int*>(smem + L.scal);            // [T] pool rows
  int* flags_s = rows_s + kMaxVerifyTokens;                       // 0 ok, 1 skip
  float* scal_f = reinterpret_cast<float*>(smem + L.scal + 68);   // [0..7] partials, [8] q.k,
                                                                  // [12..15] output-norm partials
  float* red = reinterpret_cast<float*>(smem + L.red);

  // the next launch may schedule once every CTA is resident; nothing is read before the
  // previous grid has finished
  griddep_launch_dependents();
  griddep_wait();

  // ---- rows, validation and the initial tile (copy-issuing warp) ---------------------
  if (ctrl) {
    const int r = (lane < T) ? __ldg(p.state_indices + static_cast<size_t>(b) * T + lane) : 0;
    const int na = __shfl_sync(0xffffffffu, lane == 0 ? __ldg(p.num_accepted + b) : 0, 0);
    const int r0 = __shfl_sync(0xffffffffu, r, 0);
    const bool out_of_range = lane < T && (r < 0 || r >= p.num_slots);
    const bool any_bad_row = __ballot_sync(0xffffffffu, out_of_range) != 0u;
    const int src = __shfl_sync(0xffffffffu, r, (na >= 1 && na <= T) ? na - 1 : 0);
    if (lane < T) rows_s[lane] = r;
    if (lane == 0) {
      int skip = 0;
      if (r0 < 0) {
        skip = 1;  // padding request
      } else if (any_bad_row) {
        skip = 1;
        atomic_status(p.status, GDN_STATUS_BAD_SLOT);
      } else if (na < 1 || na > T) {
        skip = 1;
        atomic_status(p.status, GDN_STATUS_BAD_LEN);
      }
      flags_s[0] = skip;
      if (!skip) {
        for (int c = 0; c < NCHUNK; ++c) mbar_init(&bars[c], 1u);
        fence_mbar_init();
        const float* tile_g = p.state + (static_cast<size_t>(src) * p.H + h) * static_cast<size_t>(D * D);
        const uint64_t pol = l2_policy_evict_first();
#pragma unroll
        for (int c = 0; c < NCHUNK; ++c) {
          mbar_arrive_expect_tx(&bars[c], CHUNK_BYTES);
          bulk_load_hint(tile + c * CHUNK_ROWS * D, tile_g + c * CHUNK_ROWS * D, CHUNK_BYTES, &bars[c], pol);
        }
      }
    }
  }

  const bool is_q = tid < D;
  const bool is_k = tid >= 128 && tid < 128 + D;
  const int ii = is_q ? tid : tid - 128;
  const int c4 = lane % VPR, rsub = lane / VPR;
  float4* tile4 = reinterpret_cast<float4*>(tile);
  bool timeout = false;

  // fused conv: thread i of the q range owns the q and v channels of key index i, thread i
  // of the k range the k channel; the window row is the request's column-0 row, read here
  // only when that row and the acceptance count are valid (the copy-issuing warp skips the
  // request otherwise, before anything is written)
  const bool conv = (fl & GDN_FUSE_CONV) != 0u;
  const bool cbf16 = (fl & GDN_QKV_BF16) != 0u;
  const int HD = p.H * D;
  const int cx = is_q ? h * D + ii : HD + h * D + ii;
  const int cv = 2 * HD + h * D + ii;
  const int CW = T + 2;
  size_t wx = 0, wv = 0;
  float sx[3] = {0.0f, 0.0f, 0.0f}, sv[3] = {0.0f, 0.0f, 0.0f};
  if (conv && !ctrl && (is_q || is_k)) {
    const int r0 = __ldg(p.state_indices + static_cast<size_t>(b) * T);
    const int na = __ldg(p.num_accepted + b);
    if (r0 >= 0 && r0 < p.num_slots && na >= 1 && na <= T) {
      wx = (static_cast<size_t>(r0) * p.channels + cx) * CW + (na - 1);
      wv = (static_cast<size_t>(r0) * p.channels + cv) * CW + (na - 1);
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        sx[j] = conv_window_load(p.conv_pool, wx + j, cbf16);
        if (is_q) sv[j] = conv_window_load(p.conv_pool, wv + j, cbf16);
      }
      wx -= (na - 1);  // row starts, for the rewrite
      wv -= (na - 1);
    }
  }

  for (int t = 0; t < T; ++t) {
    const int bt = b * T + t;  // inputs and outputs are [B][T][H][...]: position t of request b
    float* vec = reinterpret_cast<float*>(smem + L.vec) + (t & 1) * 5 * D;
    float* q_s = vec;
    float* b_s = vec;  // b takes q's place after the sums
    float* k_s = vec + D;
    float* qdec_s = vec + 2 * D;
    float* kdec_s = vec + 3 * D;
    float* dec_s = vec + 4 * D;

    // ---- position t: gates, token, decays, norm partials -----------------------------
    float x = 0.0f, vj = 0.0f, lam = 0.0f, beta = 1.0f, ga = 0.0f, gdt = 0.0f, og = 0.0f;
    if (!ctrl) {
      const int di = dlam == 1 ? 0 : ii;
      if (is_q || is_k) {
        lam = __ldg(p.lam + (static_cast<size_t>(bt) * p.H + h) * dlam + di);
        if (fl & GDN_GATE_KDA) {
          ga = __ldg(p.a_log + h);
          gdt = __ldg(p.dt_bias + static_cast<size_t>(h) * dlam + di);
        }
      }
      if ((fl & GDN_OUT_NORM_GATE) && is_q) og = __ldg(p.out_gate + (static_cast<size_t>(bt) * p.H + h) * D + ii);
      if (p.beta) beta = __ldg(p.beta + static_cast<size_t>(bt) * p.H + h);
      if (conv) {
        if (is_q || is_k) {
          const size_t xr = static_cast<size_t>(bt) * p.channels;
          x = conv_window_step(p, cx, sx, load_elem(p.mixed, xr + cx, cbf16));
          if (is_q) vj = conv_window_step(p, cv, sv, load_elem(p.mixed, xr + cv, cbf16));
        }
      } else {
        load_token(p, bt, h, 0, tid, &x, &vj);
      }
      if (fl & GDN_GATE_RAW) {
        lam = log_sigmoidf_(lam);
        if (p.beta) beta = sigmoidf_(beta);
      } else if (fl & GDN_GATE_KDA) {
        lam = p.lower_bound * sigmoidf_(expf(ga) * (lam + gdt));
        if (p.beta) beta = sigmoidf_(beta);
      }
      const float ss = warp_sum(x * x);
      if (lane == 0) scal_f[warp] = ss;
      if (is_q) {
        const float dcy = expf(lam);
        q_s[ii] = x;
        qdec_s[ii] = x * dcy;
        dec_s[ii] = dcy;
      } else if (is_k) {
        k_s[ii] = x;
        kdec_s[ii] = x * expf(lam);
      }
    }
    if (t == 0) {
      __syncthreads();  // (A) first position: also the rows, flags and barrier init
      if (ctrl || flags_s[0]) return;
    } else {
      consumer_sync();  // (A) the previous position's tile update is complete
    }

    const float qss = scal_f[0] + scal_f[1] + scal_f[2] + scal_f[3];
    const float kss = scal_f[4] + scal_f[5] + scal_f[6] + scal_f[7];
    const bool l2 = (fl & GDN_NO_QK_L2NORM) == 0u;
    const float kinv = l2 ? 1.0f / sqrtf(kss + p.l2_eps) : 1.0f;
    const float qsc = (l2 ? 1.0f / sqrtf(qss + p.l2_eps) : 1.0f) * p.q_scale;
    if (warp == NW - 1) {
      float s = 0.0f;
#pragma unroll
      for (int d = lane; d < D; d += 32) s = fmaf(q_s[d], k_s[d], s);
      s = warp_sum(s);
      if (lane == 0) scal_f[8] = s;
    }

    // ---- phase 1: r_k = S^T (e^lambda k), r_q = S^T (e^lambda q) on the raw vectors ----
    float ak[4] = {0.f, 0.f, 0.f, 0.f}, aq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) {
      if (t == 0 && !mbar_wait(&bars[c], 0u)) timeout = true;
#pragma unroll
      for (int it = c * ITC; it < (c + 1) * ITC; ++it) {
        const int r = it * RPI + warp * RPW + rsub;
        if (r < D) {
          const float4 s = tile4[r * VPR + c4];
          const float kd = kdec_s[r], qd = qdec_s[r];
          ak[0] = fmaf(s.x, kd, ak[0]);
          ak[1] = fmaf(s.y, kd, ak[1]);
          ak[2] = fmaf(s.z, kd, ak[2]);
          ak[3] = fmaf(s.w, kd, ak[3]);
          aq[0] = fmaf(s.x, qd, aq[0]);
          aq[1] = fmaf(s.y, qd, aq[1]);
          aq[2] = fmaf(s.z, qd, aq[2]);
          aq[3] = fmaf(s.w, qd, aq[3]);
        }
      }
    }
#pragma unroll
    for (int off = VPR; off < 32; off <<= 1) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        ak[m] += __shfl_xor_sync(0xffffffffu, ak[m], off);
        aq[m] += __shfl_xor_sync(0xffffffffu, aq[m], off);
      }
    }
    if (warp >= 4 && rsub == 0) {
      float* r0 = red + (warp - 4) * 2 * D + c4 * 4;
      *reinterpret_cast<float4*>(r0) = make_float4(ak[0], ak[1], ak[2], ak[3]);
      *reinterpret_cast<float4*>(r0 + D) = make_float4(aq[0], aq[1], aq[2], aq[3]);
    }
    consumer_sync();  // (D)
    if (warp < 4 && rsub == 0) {
      float* r0 = red + warp * 2 * D + c4 * 4;
      float4 pk = *reinterpret_cast<float4*>(r0), pq = *reinterpret_cast<float4*>(r0 + D);
      pk.x += ak[0];
      pk.y += ak[1];
      pk.z += ak[2];
      pk.w += ak[3];
      pq.x += aq[0];
      pq.y += aq[1];
      pq.z += aq[2];
      pq.w += aq[3];
      *reinterpret_cast<float4*>(r0) = pk;
      *reinterpret_cast<float4*>(r0 + D) = pq;
    }
    if (consumer_sync_or(timeout)) {  // (E)
      if (tid == 0) atomic_status(p.status, GDN_STATUS_TIMEOUT);
      return;
    }
    // the window keeps the last T + 2 inputs: the two after the offset, then the round's.
    // Written only past the timeout check of the first position, so a call that gave up
    // has left the window as it was (all reads of the window precede the loop).
    if (conv && (is_q || is_k)) {
      if (t == 0) {
        conv_window_store(p.conv_pool, wx, sx[0], cbf16);
        conv_window_store(p.conv_pool, wx + 1, sx[1], cbf16);
        if (is_q) {
          conv_window_store(p.conv_pool, wv, sv[0], cbf16);
          conv_window_store(p.conv_pool, wv + 1, sv[1], cbf16);
        }
      }
      conv_window_store(p.conv_pool, wx + 2 + t, sx[2], cbf16);
      if (is_q) conv_window_store(p.conv_pool, wv + 2 + t, sv[2], cbf16);
    }

    // ---- phase 2: residual, write strength, readout of position t -------------------
    float oj = 0.0f;
    if (is_q) {
      const int j = tid;
      float rk = red[j] + red[2 * D + j];
      rk += red[4 * D + j];
      rk += red[6 * D + j];
      float rq = red[D + j] + red[3 * D + j];
      rq += red[5 * D + j];
      rq += red[7 * D + j];
      rk = __fmul_rn(rk, kinv);
      rq = __fmul_rn(rq, qsc);
      const float bj = (fl & GDN_PLAIN_UPDATE) ? beta * vj : beta * (vj - rk);
      oj = fmaf(scal_f[8] * qsc * kinv, bj, rq);
      if (!(fl & GDN_OUT_NORM_GATE)) p.o[(static_cast<size_t>(bt) * p.H + h) * D + j] = oj;
      b_s[j] = bj;
    }
    if (fl & GDN_OUT_NORM_GATE) {  // KDA output epilogue, as in the decode kernel
      const float ss = warp_sum(oj * oj);
      if (lane == 0 && warp < 4) scal_f[12 + warp] = ss;
      consumer_sync();
      if (is_q) {
        const float ms = (scal_f[12] + scal_f[13] + scal_f[14] + scal_f[15]) / static_cast<float>(D);
        const float w = p.out_norm_w ? __ldg(p.out_norm_w + tid) : 1.0f;
        p.o[(static_cast<size_t>(bt) * p.H + h) * D + tid] = oj * (1.0f / sqrtf(ms + p.out_eps)) * w * sigmoidf_(og);
      }
    }
    consumer_sync();  // (F) b is in shared memory; the sums have been read

    // ---- phase 3: S <- D(lambda) S + k b^T, kept on chip and stored to row t ----------
    float* out = p.state + (static_cast<size_t>(rows_s[t]) * p.H + h) * static_cast<size_t>(D * D);
    const float4 bb = reinterpret_cast<const float4*>(b_s)[c4];
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int r = it * RPI + warp * RPW + rsub;
      if (r < D) {
        const float4 s = tile4[r * VPR + c4];
        const float dc = dec_s[r], kk = k_s[r] * kinv;
        float4 o4;
        o4.x = fmaf(kk, bb.x, dc * s.x);
        o4.y = fmaf(kk, bb.y, dc * s.y);
        o4.z = fmaf(kk, bb.z, dc * s.z);
        o4.w = fmaf(kk, bb.w, dc * s.w);
        *reinterpret_cast<float4*>(out + r * D + c4 * 4) = o4;
        tile4[r * VPR + c4] = o4;
      }
    }
  }
}

constexpr int kMaxDevices = 64;

template <int D>
cudaError_t launch_verify_d(const DecodeParams& p, cudaStream_t stream) {
  static std::atomic<int> configured[kMaxDevices];
  const VerifyLayout L = verify_layout(D);
  int dev = 0;
  cudaError_t err0 = cudaGetDevice(&dev);
  if (err0 != cudaSuccess) return err0;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    cudaError_t err = cudaFuncSetAttribute(gdn_verify_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(L.total));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(gdn_verify_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (err != cudaSuccess) return err;
    configured[dev].store(1, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.H));
  cfg.blockDim = dim3(NT_DECODE);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, gdn_verify_kernel<D>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const DecodeParams& p, cudaStream_t stream) {
  switch (p.D) {
    case 16: return launch_verify_d<16>(p, stream);
    case 32: return launch_verify_d<32>(p, stream);
    case 64: return launch_verify_d<64>(p, stream);
    case 128: return launch_verify_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
