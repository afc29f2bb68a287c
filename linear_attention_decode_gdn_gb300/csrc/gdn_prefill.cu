// gdn_prefill.cu -- the prompt through the recurrence, chunk by chunk (WY/UT form).
//
// Evolution article, "Prefill中的Chunk微观并行" (its six-step order): inside a chunk of
// C tokens with in-chunk cumulative log-decays gamma_t (per key channel),
//   A_ts = beta_t k_t^T D(gamma_t - gamma_s) k_s   (s < t),   P_ts = q_t^T D(gamma_t - gamma_s) k_s  (s <= t)
//   (I + A) B = diag(beta) (V - Ktil S0),   Ktil_t = e^{gamma_t} k_t       (the new values b_t)
//   O_t = (Qtil S0)_t + sum_{s<=t} P_ts B_s,  Qtil_t = e^{gamma_t} q_t
//   S_C = D(gamma_C) S0 + Khat^T B,          Khat_s = e^{gamma_C - gamma_s} k_s
// which reproduces, token for token, the decode step's recurrence (decay first, residual on
// the decayed state, outer-product write, post-update readout; S[dk][dv], o = S^T q).  The
// plain update (b = beta v) has no A.  One CTA owns one (request, head) and keeps its state
// in shared memory across the chunks; the products run on FP32 CUDA cores (fp32 keeps the
// state at decode precision; the state leaves for the pool row at the end: the base a
// DeltaLog decode continues from, DeltaLog notes Sec. 2.8).
#include <atomic>

#include "gdn_device.cuh"

namespace gdn {
namespace {

constexpr int PC = 32;  // tokens per chunk (one warp's width: the pair reductions map s to lanes)

struct PrefillLayout {
  uint32_t S, Kn, Qn, V, Kt, Y, A, P, gam, bet, eg, KQt, total;
};

// [Ktil; Qtil] stored transposed for the first product at head size 128: row c holds the
// 2*PC entries of key channel c, padded to a 16-byte multiple
constexpr int KQS = 2 * PC + 4;
// A is stored column-major with padded columns for the right-looking substitution
constexpr int ATS = PC + 4;

__host__ __device__ inline PrefillLayout prefill_layout(int D, int dlam) {
  PrefillLayout L{};
  uint32_t off = 0;
  L.S = off;    // state [D][D]
  off += static_cast<uint32_t>(D * D * 4);
  L.Kn = off;   // normalised keys [PC][D]
  off += static_cast<uint32_t>(PC * D * 4);
  L.Qn = off;   // normalised, scaled queries; then Qtil
  off += static_cast<uint32_t>(PC * D * 4);
  L.V = off;    // values; then R; then B
  off += static_cast<uint32_t>(PC * D * 4);
  L.Kt = off;   // Ktil; then Khat
  off += static_cast<uint32_t>(PC * D * 4);
  L.Y = off;    // Qtil S0
  off += static_cast<uint32_t>(PC * D * 4);
  L.A = off;    // column-major: A[s * ATS + t] (row t, column s), columns padded to ATS
  off += static_cast<uint32_t>(PC * ATS * 4);
  L.P = off;
  off += static_cast<uint32_t>(PC * PC * 4);
  L.gam = off;  // cumulative log-decays [PC][dlam]
  off += static_cast<uint32_t>(PC * dlam * 4);
  L.bet = off;  // [PC]
  off += static_cast<uint32_t>(PC * 4);
  L.eg = off;   // per-head decay: e^{gamma_t} [PC], then e^{gamma_C - gamma_t} [PC]
  off += static_cast<uint32_t>(2 * PC * 4);
  off = (off + 15u) & ~15u;
  L.KQt = off;  // [D][KQS] (head size 128 only)
  off += (D == 128) ? static_cast<uint32_t>(D * KQS * 4) : 0u;
  L.total = off;
  return L;
}

// Two FP32 lanes in one 64-bit register (low half first) and the packed FMA of sm_100+
// (fma.rn.f32x2): one instruction, two FMAs, each rounded as fmaf rounds.
using f2 = unsigned long long;
__device__ __forceinline__ f2 f2_splat(float x) {
  f2 r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// v[i] of every lane -> lane l holds the sum over lanes of v[l] (32 values, 31 shuffles).
__device__ __forceinline__ float transpose_reduce(float (&v)[PC], int lane) {
#pragma unroll
  for (int k = PC / 2; k >= 1; k >>= 1) {
    const bool upper = (lane & k) != 0;
#pragma unroll
    for (int i = 0; i < k; ++i) {
      const float send = upper ? v[i] : v[i + k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, k);
      v[i] = (upper ? v[i + k] : v[i]) + recv;
    }
  }
  return v[0];
}

// Width-4 causal conv + SiLU of channel ch at prompt position pos (evolution article, "去掉分母
// 引入卷积"): the four inputs pos-3 .. pos come from mixed_qkv [B][T][channels], or, before
// the prompt, from the slot's conv state (columns 0..2 = positions -3..-1).  Same product
// order as the decode kernels' one-step conv.
__device__ __forceinline__ float prefill_conv(const DecodeParams& p, int b, int slot, int pos, int ch,
                                              bool bf16) {
  const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w) + ch);
  float x[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int pj = pos - 3 + j;
    if (pj >= 0) {
      x[j] = load_elem(p.mixed, (static_cast<size_t>(b) * p.T + pj) * p.channels + ch, bf16);
    } else {
      const size_t at = (static_cast<size_t>(slot) * p.channels + ch) * 3 + (pj + 3);
      x[j] = bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(p.conv_pool)[at])
                  : static_cast<const float*>(p.conv_pool)[at];
    }
  }
  float acc = x[0] * w.x;
  acc = fmaf(x[1], w.y, acc);
  acc = fmaf(x[2], w.z, acc);
  acc = fmaf(x[3], w.w, acc);
  if (p.conv_b != nullptr) acc += __ldg(p.conv_b + ch);
  return siluf_(acc);
}

// EXT instances carry the fused conv, the KDA gate parametrisation and the output
// epilogue; the others compile them out.  At head size 128 shared memory admits one CTA
// per SM, so the register budget is the whole 255; smaller heads keep two CTAs per SM.
template <int D, bool EXT>
__global__ void __launch_bounds__(NT, D == 128 ? 1 : 2) gdn_prefill_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int TCOL = D / 16;  // product tiles: 16 x 16 thread grid
  constexpr int NI = (D + 31) / 32;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / p.H;
  const int h = blockIdx.x - b * p.H;
  const int dlam = p.dlam;
  const uint32_t fl = p.flags;
  const bool bf16 = (fl & GDN_QKV_BF16) != 0u;
  const bool plain = (fl & GDN_PLAIN_UPDATE) != 0u;
  const bool l2 = (fl & GDN_NO_QK_L2NORM) == 0u;
  const bool conv = EXT && (fl & GDN_FUSE_CONV) != 0u;
  const bool kda_gate = EXT && (fl & GDN_GATE_KDA) != 0u;
  const bool epilogue = EXT && (fl & GDN_OUT_NORM_GATE) != 0u;
  const int T = p.T;
  const int HD = p.H * D;

  griddep_launch_dependents();
  griddep_wait();

  const int slot = __ldg(p.slot + b);
  if (slot < 0) return;  // padding request
  if (slot >= p.num_slots) {
    if (tid == 0) atomic_status(p.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  const int n_tok = p.seq_lens ? __ldg(p.seq_lens + b) : T;
  if (n_tok < 0 || n_tok > T) {
    if (tid == 0) atomic_status(p.status, GDN_STATUS_BAD_LEN);
    return;
  }

  const PrefillLayout L = prefill_layout(D, dlam);
  float* S = reinterpret_cast<float*>(smem + L.S);
  float* Kn = reinterpret_cast<float*>(smem + L.Kn);
  float* Qn = reinterpret_cast<float*>(smem + L.Qn);
  float* V = reinterpret_cast<float*>(smem + L.V);
  float* Kt = reinterpret_cast<float*>(smem + L.Kt);
  float* Y = reinterpret_cast<float*>(smem + L.Y);
  float* A = reinterpret_cast<float*>(smem + L.A);
  float* P = reinterpret_cast<float*>(smem + L.P);
  float* gam = reinterpret_cast<float*>(smem + L.gam);
  float* bet = reinterpret_cast<float*>(smem + L.bet);
  float* eg = reinterpret_cast<float*>(smem + L.eg);
  float* ek = eg + PC;
  float* KQt = reinterpret_cast<float*>(smem + L.KQt);

  float* Sg = p.state + (static_cast<size_t>(slot) * p.H + h) * static_cast<size_t>(D * D);
  for (int i = tid; i < D * D / 4; i += NT)
    reinterpret_cast<float4*>(S)[i] = reinterpret_cast<const float4*>(Sg)[i];

  const int rg = tid >> 4, cg = tid & 15;  // product tile coordinates

  for (int t0 = 0; t0 < n_tok; t0 += PC) {
    const int n = (n_tok - t0 < PC) ? n_tok - t0 : PC;
    __syncthreads();  // the previous chunk is done with every buffer

    // ---- tokens: one warp per token; per-token L2 norms; positions >= n are zero --------
    // every load of the warp's tokens is issued before any is used, so the chunk waits for
    // one round trip rather than one per token
    {
      constexpr int TPW = PC / NW;  // tokens per warp
      float qv[TPW][NI], kv[TPW][NI], vv[TPW][NI], lv[TPW][NI], bv[TPW];
      if (conv) {
#pragma unroll
        for (int u = 0; u < TPW; ++u) {
          const int tt = warp + NW * u;
          const bool live = tt < n;
          const size_t tokrow = (static_cast<size_t>(b) * T + t0 + tt) * p.H + h;
#pragma unroll
          for (int i = 0; i < NI; ++i) {
            const int c = lane + 32 * i;
            qv[u][i] = kv[u][i] = vv[u][i] = lv[u][i] = 0.0f;
            if (live && c < D) {
              qv[u][i] = prefill_conv(p, b, slot, t0 + tt, h * D + c, bf16);
              kv[u][i] = prefill_conv(p, b, slot, t0 + tt, HD + h * D + c, bf16);
              vv[u][i] = prefill_conv(p, b, slot, t0 + tt, 2 * HD + h * D + c, bf16);
            }
            if (live && c < dlam) lv[u][i] = __ldg(p.lam + tokrow * dlam + c);
          }
          bv[u] = live ? (p.beta ? __ldg(p.beta + tokrow) : 1.0f) : 0.0f;
        }
      } else {
      // raw loads first (the dtype branch outside the loops), conversions after them
      uint32_t qr[TPW][NI], kr[TPW][NI], vr[TPW][NI];
#pragma unroll
      for (int u = 0; u < TPW; ++u) {
        const int tt = warp + NW * u;
        const bool live = tt < n;
        const size_t tokrow = (static_cast<size_t>(b) * T + t0 + tt) * p.H + h;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const int c = lane + 32 * i;
          qr[u][i] = kr[u][i] = vr[u][i] = 0u;
          lv[u][i] = 0.0f;
          if (live && c < D) {
            const size_t at = tokrow * D + c;
            if (bf16) {
              qr[u][i] = __ldg(static_cast<const uint16_t*>(p.q) + at);
              kr[u][i] = __ldg(static_cast<const uint16_t*>(p.k) + at);
              vr[u][i] = __ldg(static_cast<const uint16_t*>(p.v) + at);
            } else {
              qr[u][i] = __float_as_uint(__ldg(static_cast<const float*>(p.q) + at));
              kr[u][i] = __float_as_uint(__ldg(static_cast<const float*>(p.k) + at));
              vr[u][i] = __float_as_uint(__ldg(static_cast<const float*>(p.v) + at));
            }
          }
          if (live && c < dlam) lv[u][i] = __ldg(p.lam + tokrow * dlam + c);
        }
        bv[u] = live ? (p.beta ? __ldg(p.beta + tokrow) : 1.0f) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < TPW; ++u)
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          qv[u][i] = bf16 ? __uint_as_float(qr[u][i] << 16) : __uint_as_float(qr[u][i]);
          kv[u][i] = bf16 ? __uint_as_float(kr[u][i] << 16) : __uint_as_float(kr[u][i]);
          vv[u][i] = bf16 ? __uint_as_float(vr[u][i] << 16) : __uint_as_float(vr[u][i]);
        }
      }
#pragma unroll
      for (int u = 0; u < TPW; ++u) {
        const int tt = warp + NW * u;
        float sq = 0.0f, sk = 0.0f;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          sq = fmaf(qv[u][i], qv[u][i], sq);
          sk = fmaf(kv[u][i], kv[u][i], sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        // one reciprocal square root per vector (a few ulp; the decode kernels' exact
        // sqrt-and-divide would cost most of this stage)
        const float qsc = (l2 ? rsqrtf(sq + p.l2_eps) : 1.0f) * p.q_scale;
        const float kinv = l2 ? rsqrtf(sk + p.l2_eps) : 1.0f;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const int c = lane + 32 * i;
          if (c < D) {
            const float qn = qv[u][i] * qsc, kn = kv[u][i] * kinv;
            Qn[tt * D + c] = qn;
            Kn[tt * D + c] = kn;
            V[tt * D + c] = vv[u][i];
            if (D == 128 && dlam == 1) {  // channel-major copies: pair sums, then Ktil / Qtil
              KQt[c * KQS + tt] = kn;
              KQt[c * KQS + PC + tt] = qn;
            }
          }
          if (c < dlam) gam[tt * dlam + c] = lv[u][i];  // gate inputs; transformed below
        }
        if (lane == 0) bet[tt] = bv[u];
      }
    }
    __syncthreads();

    // ---- gate parametrisations, once per element (kept out of the unrolled token code) --
    if (fl & (GDN_GATE_RAW | GDN_GATE_KDA)) {
      const float ga = kda_gate ? expf(__ldg(p.a_log + h)) : 0.0f;
      for (int idx = tid; idx < n * dlam; idx += NT) {  // live tokens only
        const int c = idx - (idx / dlam) * dlam;
        const float x = gam[idx];
        gam[idx] = kda_gate ? p.lower_bound * sigmoidf_(ga * (x + __ldg(p.dt_bias + static_cast<size_t>(h) * dlam + c)))
                            : log_sigmoidf_(x);
      }
      if (p.beta)
        for (int tt = tid; tt < n; tt += NT) bet[tt] = sigmoidf_(bet[tt]);
      __syncthreads();
    }

    // ---- cumulative log-decays inside the chunk --------------------------------------
    // Per-key decay: the pair factor e^{gamma_t - gamma_s} is split at a reference token
    // (evolution article, appendix 1 "chunk内 A和M 的计算": 16-token sub-blocks; rows of
    // sub-block a and columns before it use a's first token, both exponents <= 0; the
    // diagonal sub-blocks use their own first token, the column exponent then spans at most
    // 15 tokens).  Here ref(t) = 0 for t < 16, else 16, and a column s < 16 carries both
    // references.  The split needs every factor's exponent <= 80 (no fp32 overflow); the
    // pages bound it through lower_bound = -5, which this interface does not assume, so
    // it is checked per chunk and the exact per-term form is used where it fails.
    bool split_ok = true;
    for (int c = tid; c < dlam; c += NT) {
      // all 32 loads first, then the running sum in registers (no load-store chain)
      float g[PC];
#pragma unroll
      for (int tt = 0; tt < PC; ++tt) g[tt] = gam[tt * dlam + c];
#pragma unroll
      for (int tt = 1; tt < PC; ++tt) g[tt] += g[tt - 1];
#pragma unroll
      for (int tt = 0; tt < PC; ++tt) gam[tt * dlam + c] = g[tt];
      if (dlam > 1) {
#pragma unroll
        for (int tt = 0; tt < PC; ++tt) {
          const float e_row = g[tt] - (tt < 16 ? g[0] : g[16]);
          const float e_col = fmaxf(g[16] - g[tt], tt < 16 ? g[0] - g[tt] : -INFINITY);
          if (!(fmaxf(e_row, e_col) <= 80.0f)) split_ok = false;  // also catches NaN
        }
      }
    }
    const bool split = (dlam > 1) && !__syncthreads_or(!split_ok);
    // per-head decay: its 32 distinct factors e^{gamma_t} and e^{gamma_C - gamma_t}, once (read
    // after the barrier that ends the pair sums)
    if (dlam == 1 && warp == 0) {
      eg[lane] = expf(gam[lane]);
      ek[lane] = expf(gam[PC - 1] - gam[lane]);
    }

    // column factors of the split: Km16[s][c] = k_s[c] e^{gamma_16 - gamma_s} (all s, in
    // the Khat buffer) and Km0[s][c] = k_s[c] e^{gamma_0 - gamma_s} (s < 16, in Y); both
    // buffers are free until the products below
    float* Km16 = Kt;
    float* Km0 = Y;
    if (split) {
      for (int i = tid; i < (PC + 16) * D; i += NT) {
        const int r = i / D, c = i - r * D;
        if (r < PC)
          Km16[r * D + c] = Kn[r * D + c] * expf(gam[16 * dlam + c] - gam[r * dlam + c]);
        else
          Km0[(r - PC) * D + c] = Kn[(r - PC) * D + c] * expf(gam[c] - gam[(r - PC) * dlam + c]);
      }
      __syncthreads();
    }

    // ---- A (strictly lower, times beta_t) and P (lower with the diagonal) --------------
    // warp w takes rows t = w, w + 8, ...; lane = key channel; the pair sums end in lane s
    // (a per-head decay at head size 128 uses the channel-major copies instead, below)
    if (split) {
      for (int t = warp; t < PC; t += NW) {
        float ak[PC], aq[PC];
#pragma unroll
        for (int s2 = 0; s2 < PC; ++s2) ak[s2] = aq[s2] = 0.0f;
        const float* kml = (t < 16) ? Km0 : Km16;  // columns s < 16
#pragma unroll 1
        for (int i = 0; i < NI; ++i) {
          const int c = lane + 32 * i;
          if (c < D) {
            const float f = expf(gam[t * dlam + c] - gam[(t < 16 ? 0 : 16) * dlam + c]);
            const float kt = Kn[t * D + c] * f, qt = Qn[t * D + c] * f;
#pragma unroll
            for (int s2 = 0; s2 < PC; ++s2) {
              const float w = (s2 < 16) ? kml[s2 * D + c] : Km16[s2 * D + c];
              ak[s2] = fmaf(kt, w, ak[s2]);
              aq[s2] = fmaf(qt, w, aq[s2]);
            }
          }
        }
        const float a_ts = transpose_reduce(ak, lane);
        const float p_ts = transpose_reduce(aq, lane);
        A[lane * ATS + t] = (lane < t) ? bet[t] * a_ts : 0.0f;
        P[t * PC + lane] = (lane <= t) ? p_ts : 0.0f;
      }
    } else if (D == 128 && dlam == 1) {
      // per-head decay on the channel-major copies: warp w takes rows 4w .. 4w+3, lane s the
      // column; per channel one broadcast float4 of k_t, one of q_t and k_s of the lane, and
      // no reduction across lanes
      const int tr = warp * 4;
      float aa[4] = {0.0f, 0.0f, 0.0f, 0.0f}, ap[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 8
      for (int c = 0; c < D; ++c) {
        const float4 kt = *reinterpret_cast<const float4*>(KQt + c * KQS + tr);
        const float4 qt = *reinterpret_cast<const float4*>(KQt + c * KQS + PC + tr);
        const float ks = KQt[c * KQS + lane];
        aa[0] = fmaf(kt.x, ks, aa[0]);
        aa[1] = fmaf(kt.y, ks, aa[1]);
        aa[2] = fmaf(kt.z, ks, aa[2]);
        aa[3] = fmaf(kt.w, ks, aa[3]);
        ap[0] = fmaf(qt.x, ks, ap[0]);
        ap[1] = fmaf(qt.y, ks, ap[1]);
        ap[2] = fmaf(qt.z, ks, ap[2]);
        ap[3] = fmaf(qt.w, ks, ap[3]);
      }
      float av[4];
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        const int t = tr + r4;
        const float r = expf(gam[t] - gam[lane]);  // per-head decay ratio
        av[r4] = (lane < t) ? bet[t] * (aa[r4] * r) : 0.0f;
        P[t * PC + lane] = (lane <= t) ? ap[r4] * r : 0.0f;
      }
      *reinterpret_cast<float4*>(A + lane * ATS + tr) = make_float4(av[0], av[1], av[2], av[3]);
    } else
    for (int t = warp; t < PC; t += NW) {
      float ak[PC], aq[PC];
#pragma unroll
      for (int s = 0; s < PC; ++s) ak[s] = aq[s] = 0.0f;
      if (dlam > 1) {  // exact per-term decay factors
#pragma unroll 1
        for (int i = 0; i < NI; ++i) {
          const int c = lane + 32 * i;
          if (c < D) {
            const float kt = Kn[t * D + c], qt = Qn[t * D + c];
            const float gt = gam[t * dlam + c];
#pragma unroll
            for (int s = 0; s < PC; ++s) {
              const float w = expf(gt - gam[s * dlam + c]) * Kn[s * D + c];
              ak[s] = fmaf(kt, w, ak[s]);
              aq[s] = fmaf(qt, w, aq[s]);
            }
          }
        }
      } else {  // per-head decay: plain dot products, the ratio is applied below
#pragma unroll 1
        for (int i = 0; i < NI; ++i) {
          const int c = lane + 32 * i;
          if (c < D) {
            const float kt = Kn[t * D + c], qt = Qn[t * D + c];
#pragma unroll
            for (int s = 0; s < PC; ++s) {
              const float ks = Kn[s * D + c];
              ak[s] = fmaf(kt, ks, ak[s]);
              aq[s] = fmaf(qt, ks, aq[s]);
            }
          }
        }
      }
      const float a_ts = transpose_reduce(ak, lane);
      const float p_ts = transpose_reduce(aq, lane);
      const float r = (dlam == 1) ? expf(gam[t] - gam[lane]) : 1.0f;  // per-head decay ratio
      A[lane * ATS + t] = (lane < t) ? bet[t] * (a_ts * r) : 0.0f;
      P[t * PC + lane] = (lane <= t) ? p_ts * r : 0.0f;
    }
    __syncthreads();

    // ---- Ktil = e^{gamma} k, Qtil = e^{gamma} q ----------------------------------------
    if constexpr (D == 128) {
      // KQt[c][t] = Ktil_t[c], KQt[c][PC + t] = Qtil_t[c]
      if (dlam == 1) {  // in place on the channel-major copies
        for (int i = tid; i < 2 * PC * D; i += NT) {
          const int c = i / (2 * PC), col = i - c * (2 * PC);
          KQt[c * KQS + col] *= eg[col & (PC - 1)];
        }
      } else {          // transposed from the row-major tiles
        for (int i = tid; i < PC * D; i += NT) {
          const int tt = i / D, c = i - tt * D;
          const float e = expf(gam[tt * dlam + c]);
          KQt[c * KQS + tt] = Kn[i] * e;
          KQt[c * KQS + PC + tt] = Qn[i] * e;
        }
      }
    } else {
      for (int i = tid; i < PC * D; i += NT) {
        const int tt = i / D, c = i - tt * D;
        const float e = (dlam > 1) ? expf(gam[tt * dlam + c]) : eg[tt];
        Kt[i] = Kn[i] * e;
        Qn[i] *= e;
      }
    }
    __syncthreads();

    // ---- [Ktil; Qtil] S0: R = diag(beta)(V - Ktil S0), Y = Qtil S0 ---------------------
    // the Ktil rows are skipped under the plain update
    if constexpr (D == 128) {
      // warp w: rows 16*(w/2) .. +16 of the 64, columns 64*(w%2) .. +64; lane: 4 rows and
      // two runs of 4 columns, 32 apart.  Per channel a warp loads one float4 of KQt (4
      // distinct, broadcast) and two of S (8 distinct, contiguous): 3 shared-memory
      // wavefronts per 32 FMAs per lane
      const int wb = warp >> 1, rgl = lane >> 3;
      const int row0 = wb * 16 + rgl * 4;
      const int col0 = (warp & 1) * 64 + (lane & 7) * 4;
      if (!plain || wb >= 2) {
        f2 acc2[4][4];  // [row][column pair]: columns col0 + {0,1}, {2,3}, 32 + {0,1}, 32 + {2,3}
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc2[i][j] = 0ull;
#pragma unroll 16
        for (int c = 0; c < D; ++c) {
          const float4 a = *reinterpret_cast<const float4*>(KQt + c * KQS + row0);
          const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(S + c * D + col0);
          const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(S + c * D + col0 + 32);
          const float av[4] = {a.x, a.y, a.z, a.w};
          const f2 bv[4] = {b0.x, b0.y, b1.x, b1.y};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const f2 a2 = f2_splat(av[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) acc2[i][j] = f2_fma(a2, bv[j], acc2[i][j]);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = row0 + i;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int col = col0 + 32 * hf;
            float ac[4];
            f2_unpack(acc2[i][2 * hf], ac[0], ac[1]);
            f2_unpack(acc2[i][2 * hf + 1], ac[2], ac[3]);
            if (row < PC) {
              float4 x = *reinterpret_cast<const float4*>(V + row * D + col);
              const float be = bet[row];
              x.x = be * (x.x - ac[0]);
              x.y = be * (x.y - ac[1]);
              x.z = be * (x.z - ac[2]);
              x.w = be * (x.w - ac[3]);
              *reinterpret_cast<float4*>(V + row * D + col) = x;
            } else {
              *reinterpret_cast<float4*>(Y + (row - PC) * D + col) = make_float4(ac[0], ac[1], ac[2], ac[3]);
            }
          }
        }
      }
    } else if (!plain || rg >= 8) {
      // 64 rows (16 groups of 4) x D columns (16 groups of D/16)
      const float* Ain = (rg < 8) ? Kt : Qn;
      const int r0 = (rg & 7) * 4;
      float acc[4][TCOL];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < TCOL; ++j) acc[i][j] = 0.0f;
#pragma unroll 4
      for (int c = 0; c < D; ++c) {
        float a[4], bv[TCOL];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = Ain[(r0 + i) * D + c];
#pragma unroll
        for (int j = 0; j < TCOL; ++j) bv[j] = S[c * D + cg * TCOL + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < TCOL; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tt = r0 + i;
#pragma unroll
        for (int j = 0; j < TCOL; ++j) {
          const int col = cg * TCOL + j;
          if (rg < 8)
            V[tt * D + col] = bet[tt] * (V[tt * D + col] - acc[i][j]);
          else
            Y[tt * D + col] = acc[i][j];
        }
      }
    }
    if (plain) {  // B = diag(beta) V
      for (int i = tid; i < PC * D; i += NT) V[i] *= bet[i / D];
    }
    __syncthreads();

    // ---- (I + A) B = R by forward substitution (column-parallel), then the readout -------
    // (a register-tiled product over every thread at head size 128, after the barrier)
    if (tid < D) {
      const int j = tid;
      // right-looking: once row s is final it is folded into every later row at once, so
      // each step has up to 31 independent FMAs and the chain from row to row is one FMA
      float bc[PC];
#pragma unroll
      for (int t = 0; t < PC; ++t) bc[t] = V[t * D + j];
      if (!plain) {
#pragma unroll
        for (int s = 0; s < PC - 1; ++s) {
          const float bs = bc[s];
#pragma unroll
          for (int t = s + 1; t < PC; ++t) bc[t] = fmaf(-A[s * ATS + t], bs, bc[t]);
        }
      }
      if constexpr (D == 128) {
#pragma unroll
        for (int t = 0; t < PC; ++t) V[t * D + j] = bc[t];  // B; the readout follows below
      } else {
#pragma unroll
      for (int t = 0; t < PC; ++t) {
        V[t * D + j] = bc[t];  // B for the state update
        float y[4] = {Y[t * D + j], 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int s = 0; s <= t; ++s) y[s & 3] = fmaf(P[t * PC + s], bc[s], y[s & 3]);
        const float ot = (y[0] + y[1]) + (y[2] + y[3]);
        if (epilogue)
          Y[t * D + j] = ot;  // normalised and gated below, once the whole row is known
        else if (t < n)
          p.o[((static_cast<size_t>(b) * T + t0 + t) * p.H + h) * D + j] = ot;
      }
      }
    }
    // Khat = e^{gamma_C - gamma_s} k_s (rows past n hold zero keys)
    for (int i = tid; i < PC * D; i += NT) {
      const int tt = i / D, c = i - tt * D;
      const int gc = (dlam > 1) ? c : 0;
      Kt[i] = Kn[i] * ((dlam > 1) ? expf(gam[(PC - 1) * dlam + gc] - gam[tt * dlam + gc]) : ek[tt]);
    }
    __syncthreads();

    if constexpr (D == 128) {
      // readout O = Y + P B over every thread (warp: 4 rows, lane: 4 columns)
      const int r0 = warp * 4, c0 = lane * 4;
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 y = *reinterpret_cast<const float4*>(Y + (r0 + i) * D + c0);
        acc[i][0] = y.x;
        acc[i][1] = y.y;
        acc[i][2] = y.z;
        acc[i][3] = y.w;
      }
#pragma unroll 4
      for (int s2 = 0; s2 < PC; ++s2) {
        const float4 bv = *reinterpret_cast<const float4*>(V + s2 * D + c0);
        const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float pv = P[(r0 + i) * PC + s2];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(pv, bb[jj], acc[i][jj]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = r0 + i;
        if (epilogue) {
          *reinterpret_cast<float4*>(Y + t * D + c0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        } else if (t < n) {
          float* orow = p.o + ((static_cast<size_t>(b) * T + t0 + t) * p.H + h) * D + c0;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) orow[jj] = acc[i][jj];
        }
      }
      if (epilogue) __syncthreads();  // the epilogue reads whole rows of Y
    }

    // ---- KDA output epilogue: o <- o / sqrt(mean(o^2) + eps) * w * sigmoid(g) per row ---
    if (epilogue) {
      for (int t = warp; t < n; t += NW) {
        float ss = 0.0f;
        for (int j = lane; j < D; j += 32) ss = fmaf(Y[t * D + j], Y[t * D + j], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + p.out_eps);
        const size_t orow = ((static_cast<size_t>(b) * T + t0 + t) * p.H + h) * D;
        for (int j = lane; j < D; j += 32) {
          const float w = p.out_norm_w ? __ldg(p.out_norm_w + j) : 1.0f;
          p.o[orow + j] = Y[t * D + j] * inv * w * sigmoidf_(__ldg(p.out_gate + orow + j));
        }
      }
    }

    // ---- S <- D(gamma_C) S + Khat^T B ---------------------------------------------------
    if constexpr (D == 128) {
      // lane: rows 8*rg .. +8, columns 4*cg .. +4 and 64 + 4*cg .. +4 (contiguous float4 runs
      // across the 16 lanes of a row group, for the operand loads and the state update)
      f2 acc2[8][4];  // [row][column pair]: columns 4cg + {0,1}, {2,3}, 64 + 4cg + {0,1}, {2,3}
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc2[i][j] = 0ull;
#pragma unroll 8
      for (int s = 0; s < PC; ++s) {
        const float4 a0 = *reinterpret_cast<const float4*>(Kt + s * D + rg * 8);
        const float4 a1 = *reinterpret_cast<const float4*>(Kt + s * D + rg * 8 + 4);
        const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(V + s * D + cg * 4);
        const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(V + s * D + 64 + cg * 4);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const f2 bv[4] = {b0.x, b0.y, b1.x, b1.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const f2 a2 = f2_splat(av[i]);
#pragma unroll
          for (int j = 0; j < 4; ++j) acc2[i][j] = f2_fma(a2, bv[j], acc2[i][j]);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rg * 8 + i;
        const float dC = (dlam > 1) ? expf(gam[(PC - 1) * dlam + r]) : eg[PC - 1];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float* sp = S + r * D + 64 * hf + cg * 4;
          float ac[4];
          f2_unpack(acc2[i][2 * hf], ac[0], ac[1]);
          f2_unpack(acc2[i][2 * hf + 1], ac[2], ac[3]);
          float4 x = *reinterpret_cast<const float4*>(sp);
          x.x = fmaf(dC, x.x, ac[0]);
          x.y = fmaf(dC, x.y, ac[1]);
          x.z = fmaf(dC, x.z, ac[2]);
          x.w = fmaf(dC, x.w, ac[3]);
          *reinterpret_cast<float4*>(sp) = x;
        }
      }
    } else {
      float acc[TCOL][TCOL];
#pragma unroll
      for (int i = 0; i < TCOL; ++i)
#pragma unroll
        for (int j = 0; j < TCOL; ++j) acc[i][j] = 0.0f;
#pragma unroll 4
      for (int s = 0; s < PC; ++s) {
        float a[TCOL], bv[TCOL];
#pragma unroll
        for (int i = 0; i < TCOL; ++i) a[i] = Kt[s * D + rg * TCOL + i];
#pragma unroll
        for (int j = 0; j < TCOL; ++j) bv[j] = V[s * D + cg * TCOL + j];
#pragma unroll
        for (int i = 0; i < TCOL; ++i)
#pragma unroll
          for (int j = 0; j < TCOL; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < TCOL; ++i) {
        const int r = rg * TCOL + i;
        const float dC = (dlam > 1) ? expf(gam[(PC - 1) * dlam + r]) : eg[PC - 1];
#pragma unroll
        for (int j = 0; j < TCOL; ++j) {
          const int col = cg * TCOL + j;
          S[r * D + col] = fmaf(dC, S[r * D + col], acc[i][j]);
        }
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < D * D / 4; i += NT)
    reinterpret_cast<float4*>(Sg)[i] = reinterpret_cast<const float4*>(S)[i];
  // the slot's conv state keeps the last three inputs of (old state, prompt), bit-exact;
  // every read of the old state lies before the barrier above
  if (conv && n_tok > 0) {
    for (int idx = tid; idx < 3 * D; idx += NT) {
      const int g = idx / D, c = idx - g * D;
      const int ch = g * HD + h * D + c;
      const size_t srow = (static_cast<size_t>(slot) * p.channels + ch) * 3;
      uint32_t nb[3];
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int pj = n_tok - 3 + j;
        if (pj >= 0) {
          const size_t at = (static_cast<size_t>(b) * T + pj) * p.channels + ch;
          nb[j] = bf16 ? static_cast<uint32_t>(__ldg(static_cast<const uint16_t*>(p.mixed) + at))
                       : __float_as_uint(__ldg(static_cast<const float*>(p.mixed) + at));
        } else {
          nb[j] = bf16 ? static_cast<uint32_t>(static_cast<const uint16_t*>(p.conv_pool)[srow + pj + 3])
                       : __float_as_uint(static_cast<const float*>(p.conv_pool)[srow + pj + 3]);
        }
      }
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        if (bf16)
          static_cast<uint16_t*>(p.conv_pool)[srow + j] = static_cast<uint16_t>(nb[j]);
        else
          static_cast<float*>(p.conv_pool)[srow + j] = __uint_as_float(nb[j]);
      }
    }
  }
}

constexpr int kMaxDevices = 64;

template <int D, bool EXT>
cudaError_t launch_prefill_de(const DecodeParams& p, cudaStream_t stream) {
  static std::atomic<uint32_t> configured[kMaxDevices];
  const PrefillLayout L = prefill_layout(D, p.dlam);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (configured[dev].load(std::memory_order_relaxed) < L.total) {
    err = cudaFuncSetAttribute(gdn_prefill_kernel<D, EXT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(L.total));
    if (err != cudaSuccess) return err;
    configured[dev].store(L.total, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.H));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, gdn_prefill_kernel<D, EXT>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_prefill_d(const DecodeParams& p, cudaStream_t stream) {
  if (p.flags & (GDN_FUSE_CONV | GDN_GATE_KDA | GDN_OUT_NORM_GATE)) return launch_prefill_de<D, true>(p, stream);
  return launch_prefill_de<D, false>(p, stream);
}

}  // namespace

size_t prefill_smem_bytes(int D, int dlam) { return prefill_layout(D, dlam).total; }

cudaError_t launch_prefill(const DecodeParams& p, cudaStream_t stream) {
  if (prefill_tc_supported(p)) return launch_prefill_tc(p, stream);
  if (prefill_tc_pk_supported(p)) return launch_prefill_tc_pk(p, stream);
  switch (p.D) {
    case 16: return launch_prefill_d<16>(p, stream);
    case 32: return launch_prefill_d<32>(p, stream);
    case 64: return launch_prefill_d<64>(p, stream);
    case 128: return launch_prefill_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
