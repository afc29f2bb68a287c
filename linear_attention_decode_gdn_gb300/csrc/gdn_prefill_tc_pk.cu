// gdn_prefill_tc_pk.cu -- chunked prefill on the tcgen05 tensor cores for a per-key-channel
// decay (KDA's log decay lambda_t[c]), head size 128, bf16 q/k/v.
//
// Evolution article, "Prefill中的Chunk微观并行" ("完整计算顺序"), with the decay per key channel:
// inside a chunk of C = 32 tokens with cumulative log-decays gamma_t[c],
//   Ktil_t = e^{gamma_t} (.) k_t,  Qtil_t = e^{gamma_t} (.) q_t,  Kbar_s = e^{-gamma_s} (.) k_s
//   A_ts = beta_t Ktil_t . Kbar_s  (s < t),   P_ts = Qtil_t . Kbar_s  (s <= t)
//   (I + A) B = diag(beta) (V - Ktil S0),   O = Qtil S0 + P B
//   S_C = D(gamma_C) S0 + Khat^T B,         Khat_s = e^{gamma_C - gamma_s} (.) k_s
// (k and q L2-normalised, q scaled), the same recurrence as the decode step with a per-key
// decay, token for token.  The per-channel factors go into the operands, so every product is
// a plain matrix product on the tensor cores (kind::tf32, three-term TF32 splitting as in
// gdn_prefill_tc.cu): pair sums [Ktil; Qtil] Kbar^T (M = 64, N = 32, K = 128), state read
// S^T [Ktil; Qtil]^T, state write S^T += B^T Khat, readout O^T = O^T + B^T P^T.
//
// The operand factors use the fast exponential (__expf: a few parts in 10^6 at |gamma| <= 80,
// far inside the fp32-accuracy bar of the products; 8% of the kernel's time against expf).
//
// Kbar needs e^{-gamma_s} finite: a chunk whose cumulative decay falls below e^{-80} in some
// channel forms its pair sums on the CUDA cores instead, term by term with e^{gamma_t -
// gamma_s} (exact, slow, and only for such extreme decays; the other products are unchanged).
//
// The state lives in tensor memory for the whole prompt as in gdn_prefill_tc.cu; its decay
// by D(gamma_C) is a per-column pass over TMEM (column c = key channel).  The token rows of a
// chunk (q, k, v bf16 and the fp32 log decays) arrive by 3-D TMA into swizzled staging, and
// each tensor's copy for the next chunk is issued as soon as this chunk has finished with it:
// q after the token stage, k and the decays after the Khat tile is built, v after the
// residuals (which read it from the staging, so no V tile is kept).
#include <atomic>

#include "gdn_tc.cuh"
#include "gdn_tmap.h"

namespace gdn {
namespace {

constexpr int TD = 128;      // head size of this kernel
constexpr int TC_C = 32;     // tokens per chunk
constexpr int TC_NT = 288;   // threads per CTA: 8 compute warps and the MMA-issuing warp
constexpr int ISSUER = 8;    // the warp that issues every MMA and TMA copy
constexpr int TC_ATS = TC_C + 4;

// Operand tiles (K-major, no swizzle; element (r, k) at (r/8)*128 + (k/4)*LBO + (r%8)*16 + (k%4)*4).
constexpr uint32_t X_LBO = (2 * TC_C / 8) * 128;   // [Ktil; Qtil]: 64 x 128   (1024)
constexpr uint32_t N_LBO = (TC_C / 8) * 128;       // Kbar:         32 x 128   (512)
constexpr uint32_t T128_LBO = (TD / 8) * 128;      // Khat^T, B^T:  128 x 32   (2048)
constexpr uint32_t P_LBO = (TC_C / 8) * 128;       // P:            32 x 32    (512)
constexpr uint32_t SBO = 128;

// Staging, one chunk ahead, as 128-byte column boxes of 32 rows with the 128-byte swizzle
// (16-byte chunk c of row t at position c ^ (t % 8)): q, k, v bf16 (2 boxes each), the log
// decays fp32 (4 boxes).  After the scan the decay boxes hold gamma_t[c] in place.
constexpr uint32_t ST_BOX = TC_C * 128;

// shared-memory layout (bytes)
constexpr uint32_t OFF_XH = 0;                             // [Ktil; Qtil] hi 64 x 128
constexpr uint32_t OFF_XL = OFF_XH + 2 * TC_C * TD * 4;
constexpr uint32_t OFF_NH = OFF_XL + 2 * TC_C * TD * 4;    // Kbar hi 32 x 128
constexpr uint32_t OFF_NL = OFF_NH + TC_C * TD * 4;
constexpr uint32_t OFF_KH = OFF_NL + TC_C * TD * 4;        // Khat^T hi 128 x 32
constexpr uint32_t OFF_KL = OFF_KH + TD * TC_C * 4;
constexpr uint32_t OFF_BH = OFF_KL + TD * TC_C * 4;        // B^T hi 128 x 32
constexpr uint32_t OFF_BL = OFF_BH + TD * TC_C * 4;
constexpr uint32_t OFF_PH = OFF_BL + TD * TC_C * 4;        // P hi 32 x 32
constexpr uint32_t OFF_PL = OFF_PH + TC_C * TC_C * 4;
constexpr uint32_t OFF_A = OFF_PL + TC_C * TC_C * 4;       // A column-major [s][TC_ATS]
constexpr uint32_t OFF_SQ = (OFF_A + TC_C * TC_ATS * 4 + 1023u) & ~1023u;  // staging q (1024-aligned)
constexpr uint32_t OFF_SK = OFF_SQ + 2 * ST_BOX;           // staging k
constexpr uint32_t OFF_SV = OFF_SK + 2 * ST_BOX;           // staging v
constexpr uint32_t OFF_SL = OFF_SV + 2 * ST_BOX;           // staging log decays / gamma
constexpr uint32_t OFF_DC = OFF_SL + 4 * ST_BOX;           // gamma_C[c], e^{gamma_C[c]}
constexpr uint32_t OFF_G = OFF_DC + 2 * TD * 4;            // beta, key scale, query scale per token
constexpr uint32_t OFF_EP = OFF_G + 3 * TC_C * 4;          // output epilogue: 4 x 32 partial sums, 32 scales
constexpr uint32_t OFF_BAR = OFF_EP + 5 * TC_C * 4;        // mbarriers: ps, p1, p2, drain, staging q, k, v
constexpr uint32_t OFF_TMEM = OFF_BAR + 8 * 8;
constexpr uint32_t PK_SMEM = OFF_TMEM + 16;

// TMEM columns (as gdn_prefill_tc.cu)
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_L = 128;
constexpr uint32_t TM_D1 = 256;
constexpr uint32_t TM_PS = 320;
constexpr uint32_t TM_D1B = 352;
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t IDESC_PS = tc::idesc_tf32(64, 32);
constexpr uint32_t IDESC_P1 = tc::idesc_tf32(128, 64);
constexpr uint32_t IDESC_P2 = tc::idesc_tf32(128, 128);
constexpr uint32_t IDESC_RO = tc::idesc_tf32(128, 32);

// a chunk whose cumulative log-decay stays above this in every channel forms Kbar = e^{-gamma} k
constexpr float GAMMA_FLOOR = -80.0f;

__device__ __forceinline__ uint32_t kmaj_off(int r, int k, uint32_t lbo) {
  return static_cast<uint32_t>((r >> 3) * SBO + (k >> 2) * lbo + (r & 7) * 16 + (k & 3) * 4);
}

__device__ __forceinline__ void store_split4(unsigned char* smem, uint32_t hi_base, uint32_t lo_base, uint32_t off,
                                             float a, float b, float c, float d) {
  const float ha = tc::tf32_hi(a), hb = tc::tf32_hi(b), hc = tc::tf32_hi(c), hd = tc::tf32_hi(d);
  *reinterpret_cast<float4*>(smem + hi_base + off) = make_float4(ha, hb, hc, hd);
  *reinterpret_cast<float4*>(smem + lo_base + off) = make_float4(a - ha, b - hb, c - hc, d - hd);
}

__device__ __forceinline__ void store_split1(unsigned char* smem, uint32_t hi_base, uint32_t lo_base, uint32_t off,
                                             float a) {
  const float ha = tc::tf32_hi(a);
  *reinterpret_cast<float*>(smem + hi_base + off) = ha;
  *reinterpret_cast<float*>(smem + lo_base + off) = a - ha;
}

// Byte address of element (t, c) of a staged tensor with `esz`-byte elements (boxes of
// 128 / esz elements, swizzled rows of 128 bytes).
__device__ __forceinline__ const unsigned char* staged_at(const unsigned char* base, int t, int c, uint32_t esz) {
  const uint32_t byte = static_cast<uint32_t>(c) * esz;
  const uint32_t inb = byte & 127u;
  return base + (byte >> 7) * ST_BOX + static_cast<uint32_t>(t) * 128u +
         ((((inb >> 4) ^ (static_cast<uint32_t>(t) & 7u)) << 4) | (inb & 15u));
}

// elements 4g .. 4g+3 of row t of a staged bf16 tensor, as float
__device__ __forceinline__ float4 staged4_bf16(const unsigned char* base, int t, int g) {
  const uint2 u = *reinterpret_cast<const uint2*>(staged_at(base, t, 4 * g, 2u));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xffff0000u));
}

struct TokenMapsPK {
  CUtensorMap q, k, v, lam;
};

// One 3-D box of a tensor map into shared memory, completion counted on `bar`; called by a
// whole warp with warp-uniform operands, one elected lane issues.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n .reg .b32 l;\n elect.sync l|e, 0xffffffff;\n"
      " @e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n}\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Named barrier over warps 4-7 (128 threads) returning the OR of `pred` over them, and the
// plain form.
__device__ __forceinline__ bool upper_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a, o;\n setp.ne.u32 a, %1, 0;\n bar.red.or.pred o, 2, 128, a;\n selp.u32 %0, 1, 0, o;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0u;
}
__device__ __forceinline__ void upper_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// v[i] of every lane -> the return value of lane l is the sum over the warp of v[l]
// (recursive halving: at each step a lane keeps half its partial sums and adds the partner's).
__device__ __forceinline__ float transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) {
    const bool upper = (lane & k) != 0;
#pragma unroll
    for (int i = 0; i < k; ++i) {
      const float send = upper ? v[i] : v[i + k];
      const float keep = upper ? v[i + k] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
    }
  }
  return v[0];
}

// Bounded wait for phase `parity` of `bar`, the same answer in every lane of the warp.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__global__ void __launch_bounds__(TC_NT, 1) gdn_prefill_tc_pk_kernel(const DecodeParams p,
                                                                     const __grid_constant__ TokenMapsPK maps) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / p.H;
  const int h = blockIdx.x - b * p.H;
  const uint32_t fl = p.flags;
  const bool plain = (fl & GDN_PLAIN_UPDATE) != 0u;
  const bool l2 = (fl & GDN_NO_QK_L2NORM) == 0u;
  const bool graw = (fl & GDN_GATE_RAW) != 0u;
  const bool kda = (fl & GDN_GATE_KDA) != 0u;          // KDA gate parametrisation of the decays
  const bool epi = (fl & GDN_OUT_NORM_GATE) != 0u;     // KDA output epilogue
  const int T = p.T;

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
  if (n_tok == 0) return;  // the state is left as it is

  float* gC = reinterpret_cast<float*>(smem + OFF_DC);  // gamma_C[c]
  float* dC = gC + TD;                                    // e^{gamma_C[c]}
  float* bet = reinterpret_cast<float*>(smem + OFF_G);
  float* skf = bet + TC_C;  // per-token key scale (1/|k|)
  float* sqf = bet + 2 * TC_C;  // per-token query scale (q_scale/|q|)
  float* A = reinterpret_cast<float*>(smem + OFF_A);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* stq = bars + 4;  // staging q of a chunk
  uint64_t* stk = bars + 5;  // staging k and the log decays
  uint64_t* stv = bars + 6;  // staging v
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
  const int wq = warp & 3;

  bool bad = false;
  if (tid == 0) {
    for (int i = 0; i < 7; ++i) mbar_init(&bars[i], 1u);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- staging copies (issuer warp) -------------------------------------------------------
  // loads issued per staging barrier; load i completes phase i & 1
  uint32_t nq = 0, nk = 0, nv = 0;
  float pf_beta = 0.0f;
  auto copy_q = [&](int t0) {
    if (warp != ISSUER) return;
    tc::expect_tx(stq, 2u * ST_BOX);
    for (int bx = 0; bx < 2; ++bx)
      tma_load_3d(smem_addr(smem + OFF_SQ + bx * ST_BOX), &maps.q, bx * 64, h, b * T + t0, stq);
    ++nq;
  };
  auto copy_k = [&](int t0) {
    if (warp != ISSUER) return;
    tc::expect_tx(stk, 6u * ST_BOX);
    for (int bx = 0; bx < 2; ++bx)
      tma_load_3d(smem_addr(smem + OFF_SK + bx * ST_BOX), &maps.k, bx * 64, h, b * T + t0, stk);
    for (int bx = 0; bx < 4; ++bx)
      tma_load_3d(smem_addr(smem + OFF_SL + bx * ST_BOX), &maps.lam, bx * 32, h, b * T + t0, stk);
    ++nk;
  };
  auto copy_v = [&](int t0) {
    if (warp != ISSUER) return;
    tc::expect_tx(stv, 2u * ST_BOX);
    for (int bx = 0; bx < 2; ++bx)
      tma_load_3d(smem_addr(smem + OFF_SV + bx * ST_BOX), &maps.v, bx * 64, h, b * T + t0, stv);
    ++nv;
  };
  auto load_beta = [&](int t0, int n) {
    if (warp == 4) {
      const size_t gi = (static_cast<size_t>(b) * T + t0 + lane) * p.H + h;
      pf_beta = lane < n ? (p.beta ? __ldg(p.beta + gi) : 1.0f) : 0.0f;
    }
  };
  copy_q(0);
  copy_k(0);
  copy_v(0);
  load_beta(0, n_tok < TC_C ? n_tok : TC_C);

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, TM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lb = tc::lane_base(warp);
  const int j = tid & (TD - 1);  // this thread's TMEM lane / value column
  const uint32_t sbase = smem_addr(smem);

  float* Sg = p.state + (static_cast<size_t>(slot) * p.H + h) * static_cast<size_t>(TD * TD);

  // ---- the state into TMEM, transposed (lane j, column c), with its TF32 remainder ------------
  if (warp < ISSUER) {
    const int c0 = 64 * (tid >> 7);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float v[16], lo[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = Sg[static_cast<size_t>(c0 + 16 * cc + k) * TD + j];
#pragma unroll
      for (int k = 0; k < 16; ++k) lo[k] = v[k] - tc::tf32_hi(v[k]);
      tc::st16(tmem + lb + TM_S + c0 + 16 * cc, v);
      tc::st16(tmem + lb + TM_L + c0 + 16 * cc, lo);
    }
    tc::wait_st();
  }

  uint32_t it = 0;       // the chunk being processed
  bool split = true;     // this chunk forms Kbar (every channel's gamma_C above the floor)

  // ---- token stage of chunk it (from the staging) -------------------------------------------
  // (1) warps 0-3, thread c = tid: the cumulative log-decays gamma_t[c] of the chunk, in place
  //     of the staged decays, gamma_C[c] and e^{gamma_C[c]}; (2) all compute warps: the norms
  //     and the [Ktil; Qtil] and Kbar tiles (warps 0-3 key rows t = 8 w + (lane & 7), channel
  //     groups g = (lane >> 3) + 4 i; warps 4-7 query rows); warp 4 the write strengths.
  //     Ends with the pair-sum MMAs issued when the chunk forms Kbar.
  auto token_stage = [&](int n) {
    bool low = false;
    if (warp < ISSUER) {
      if (!wait_warp(stq, it & 1u)) bad = true;
      if (!wait_warp(stk, it & 1u)) bad = true;
      unsigned char* sl = smem + OFF_SL;
      if (graw || kda) {
        // the gate parametrisation of every live decay, in place, on all compute warps:
        // logsigmoid (raw gates) or KDA's lambda = lower_bound sigmoid(e^{A_log[h]} (f + dt_bias[h][c]))
        const int c = tid & (TD - 1);
        const float ga = kda ? expf(__ldg(p.a_log + h)) : 0.0f;
        const float dtb = kda ? __ldg(p.dt_bias + static_cast<size_t>(h) * TD + c) : 0.0f;
        for (int t = tid >> 7; t < n; t += 2) {
          float* at = reinterpret_cast<float*>(const_cast<unsigned char*>(staged_at(sl, t, c, 4u)));
          // (KDA's sigmoid through the fast intrinsics: relative error a few parts in 10^7 also
          // where it is tiny; the log-sigmoid of raw gates keeps log1pf, which carries the
          // whole value of a decay near zero)
          *at = kda ? p.lower_bound * __fdividef(1.0f, 1.0f + __expf(-ga * (*at + dtb))) : log_sigmoidf_(*at);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");  // the compute warps
      }
      if (warp < 4) {
        float g = 0.0f;
#pragma unroll 4
        for (int t = 0; t < TC_C; ++t) {
          float* at = reinterpret_cast<float*>(const_cast<unsigned char*>(staged_at(sl, t, tid, 4u)));
          const float lam = t < n ? *at : 0.0f;
          g += lam;
          *at = g;
        }
        gC[tid] = g;
        dC[tid] = expf(g);
        low = g < GAMMA_FLOOR;
      }
      if (warp == 4) {
        float be = pf_beta;
        if ((graw || kda) && p.beta && lane < n) be = sigmoidf_(be);
        bet[lane] = be;
      }
    }
    split = !__syncthreads_or(low);  // gamma, beta visible; the chunk's choice is uniform
    if (warp < ISSUER) {
      const int t = 8 * wq + (lane & 7);
      const int g0 = lane >> 3;
      const bool live = t < n;
      const bool isk = warp < 4;
      const unsigned char* src = smem + (isk ? OFF_SK : OFF_SQ);
      float4 x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = live ? staged4_bf16(src, t, g0 + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
      float ss = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += x[i].x * x[i].x + x[i].y * x[i].y + x[i].z * x[i].z + x[i].w * x[i].w;
      ss += __shfl_xor_sync(0xffffffffu, ss, 8);
      ss += __shfl_xor_sync(0xffffffffu, ss, 16);
      const float sc = (l2 ? rsqrtf(ss + p.l2_eps) : 1.0f) * (isk ? 1.0f : p.q_scale);
      if ((lane >> 3) == 0) (isk ? skf : sqf)[t] = sc;
      const int r = isk ? t : TC_C + t;
      const unsigned char* gl = smem + OFF_SL;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = 4 * (g0 + 4 * i);
        const float4 g4 = *reinterpret_cast<const float4*>(staged_at(gl, t, c, 4u));
        const float a0 = x[i].x * sc, a1 = x[i].y * sc, a2 = x[i].z * sc, a3 = x[i].w * sc;
        store_split4(smem, OFF_XH, OFF_XL, kmaj_off(r, c, X_LBO), a0 * __expf(g4.x), a1 * __expf(g4.y), a2 * __expf(g4.z),
                     a3 * __expf(g4.w));
        if (isk && split)
          store_split4(smem, OFF_NH, OFF_NL, kmaj_off(t, c, N_LBO), a0 * __expf(-g4.x), a1 * __expf(-g4.y),
                       a2 * __expf(-g4.z), a3 * __expf(-g4.w));
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();  // tiles and scales visible; the staged q rows are free again (when split)
    tc::fence_after_sync();
    if (warp == ISSUER) {
      if (split) {
        // pair sums [Ktil; Qtil] Kbar^T (hi hi, lo hi, hi lo)
        const uint32_t xh = sbase + OFF_XH, xl = sbase + OFF_XL, nh = sbase + OFF_NH, nl = sbase + OFF_NL;
#pragma unroll 1
        for (int gidx = 0; gidx < 3; ++gidx) {
          const uint32_t a = gidx == 1 ? xl : xh, bb = gidx == 2 ? nl : nh;
#pragma unroll
          for (int i = 0; i < TD / 8; ++i)
            tc::mma_ss(tmem + TM_PS, tc::smem_desc(a + 2 * i * X_LBO, X_LBO, SBO),
                       tc::smem_desc(bb + 2 * i * N_LBO, N_LBO, SBO), IDESC_PS, (gidx | i) != 0);
        }
      }
      tc::commit(&bars[0]);  // (with no pair-sum MMAs: once the earlier MMAs are done)
    }
  };

  int t0 = 0;
  int n = n_tok < TC_C ? n_tok : TC_C;
  token_stage(n);
  int nt0 = TC_C;  // the next chunk's first position
  int nn = n_tok - nt0 < TC_C ? n_tok - nt0 : TC_C;
  if (split && nt0 < n_tok) {
    copy_q(nt0);
    load_beta(nt0, nn);
  }
  int prev_t0 = 0, prev_n = 0;

  // readout of a finished chunk from its TMEM output buffer (warps 4-7, called by all four
  // together), coalesced row stores; with the KDA epilogue each position's row is first
  // normalised by its RMS over the 128 value columns (four warps' partial sums) and gated:
  // o <- o / sqrt(mean(o^2) + eps) w sigmoid(g)
  float* ep_part = reinterpret_cast<float*>(smem + OFF_EP);
  float* ep_inv = ep_part + 4 * TC_C;
  // the output gates of the positions a store_output call writes, loaded ahead of it (the
  // output stores may alias them, so they cannot be hoisted past the stores)
  auto load_gates = [&](int ct0, int cn, float (&gv)[32]) {
    const size_t obase = ((static_cast<size_t>(b) * T + ct0) * p.H + h) * TD + j;
    const size_t tstride = static_cast<size_t>(p.H) * TD;
#pragma unroll
    for (int k = 0; k < 32; ++k) gv[k] = k < cn ? __ldg(p.out_gate + obase + k * tstride) : 0.0f;
  };
  auto store_output = [&](uint32_t d1, int ct0, int cn, const float (&gv)[32]) {
    float o[32], o1[16];
    tc::ld16(tmem + lb + d1 + TC_C, o1);
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = o1[k];
    tc::ld16(tmem + lb + d1 + TC_C + 16, o1);
#pragma unroll
    for (int k = 0; k < 16; ++k) o[16 + k] = o1[k];
    const size_t obase = ((static_cast<size_t>(b) * T + ct0) * p.H + h) * TD + j;
    const size_t tstride = static_cast<size_t>(p.H) * TD;
    if (epi) {
      float sq[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) sq[k] = o[k] * o[k];
      ep_part[(warp - 4) * TC_C + lane] = transpose_sum32(sq, lane);
      upper_sync();
      if (warp == 4) {
        const float ms = (ep_part[lane] + ep_part[TC_C + lane] + ep_part[2 * TC_C + lane] + ep_part[3 * TC_C + lane]) /
                         static_cast<float>(TD);
        ep_inv[lane] = 1.0f / sqrtf(ms + p.out_eps);
      }
      upper_sync();
      const float w = p.out_norm_w ? __ldg(p.out_norm_w + j) : 1.0f;
      // (the gate's sigmoid through the fast intrinsics: a few parts in 10^7)
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (k < cn) p.o[obase + k * tstride] = o[k] * ep_inv[k] * w * __fdividef(1.0f, 1.0f + __expf(-gv[k]));
      upper_sync();  // (the partial sums are rewritten by the next chunk's call)
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (k < cn) p.o[obase + k * tstride] = o[k];
    }
  };

  while (true) {
    const uint32_t d1 = (it & 1u) ? TM_D1B : TM_D1;
    if (it > 0) {
      // the previous chunk's state write and readout are complete
      if (!wait_warp(&bars[2], (it - 1) & 1u)) bad = true;
      tc::fence_after_sync();
      if (!bad && warp >= 4 && warp < ISSUER) {
        // TF32 remainder of the new state
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float v[16];
          tc::ld16(tmem + lb + TM_S + 16 * cc, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] -= tc::tf32_hi(v[k]);
          tc::st16(tmem + lb + TM_L + 16 * cc, v);
        }
        tc::wait_st();
      }
    }
    if (warp < 4) {
      // Khat^T tile (row c, column s): e^{gamma_C[c] - gamma_s[c]} times the normalised key,
      // from the staged raw key and gamma (their next copies wait until after S1)
      const int s = 8 * warp + (lane & 7);
      const float sk = skf[s];
      const int g0 = lane >> 3;
      const unsigned char* gl = smem + OFF_SL;
      const unsigned char* kl = smem + OFF_SK;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = 4 * (g0 + 4 * i);
        const float4 kx = s < n ? staged4_bf16(kl, s, g0 + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 g4 = *reinterpret_cast<const float4*>(staged_at(gl, s, c, 4u));
        const float4 c4 = *reinterpret_cast<const float4*>(gC + c);
        store_split1(smem, OFF_KH, OFF_KL, kmaj_off(c + 0, s, T128_LBO), kx.x * sk * __expf(c4.x - g4.x));
        store_split1(smem, OFF_KH, OFF_KL, kmaj_off(c + 1, s, T128_LBO), kx.y * sk * __expf(c4.y - g4.y));
        store_split1(smem, OFF_KH, OFF_KL, kmaj_off(c + 2, s, T128_LBO), kx.z * sk * __expf(c4.z - g4.z));
        store_split1(smem, OFF_KH, OFF_KL, kmaj_off(c + 3, s, T128_LBO), kx.w * sk * __expf(c4.w - g4.w));
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    if ((bad = __syncthreads_or(bad) != 0)) break;  // (S1)
    tc::fence_after_sync();

    if (warp == ISSUER) {
      // state read S^T [Ktil; Qtil]^T: hi(S) Xh, lo(S) Xh, hi(S) Xl
      const uint32_t xh = sbase + OFF_XH, xl = sbase + OFF_XL;
#pragma unroll 1
      for (int gidx = 0; gidx < 3; ++gidx) {
        const uint32_t a = tmem + (gidx == 1 ? TM_L : TM_S), bb = gidx == 2 ? xl : xh;
#pragma unroll
        for (int i = 0; i < TD / 8; ++i)
          tc::mma_ts(tmem + d1, a + 8 * i, tc::smem_desc(bb + 2 * i * X_LBO, X_LBO, SBO), IDESC_P1, (gidx | i) != 0);
      }
      tc::commit(&bars[1]);
      // the staged k rows and decays are free now (a chunk without Kbar still reads them below)
      if (split && nt0 < n_tok) copy_k(nt0);
    } else {
      // ---- A (strictly lower, times beta) and P (lower with the diagonal), on all eight
      // compute warps as in gdn_prefill_tc.cu: warps w and w + 4 share a TMEM lane quarter
      // (the M = 64 accumulator's rows t = 16 (w % 2) + lane, k.k for w % 4 < 2, q.k else);
      // warp group w / 4 takes source tokens 16 (w / 4) .. +15, lanes 16-31 the upper eight
      if (!wait_warp(&bars[0], it & 1u)) bad = true;
      tc::fence_after_sync();
      const int G = warp >> 2, half = lane >> 4;
      const int t = 16 * (warp & 1) + (lane & 15);
      const int sb = 16 * G + 8 * half;  // this thread's first source token
      const bool isA = (warp & 2) == 0;
      float ps[8];
      if (split) {
        float a16[16];
        tc::ld16(tmem + lb + TM_PS + 16 * G, a16);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float up = __shfl_sync(0xffffffffu, a16[8 + k], lane & 15);
          ps[k] = half ? up : a16[k];
        }
      } else {
        // the exact per-term pair sums: sum_c x_t[c] k_s[c] e^{gamma_t[c] - gamma_s[c]} with x
        // the normalised key (A) or query (P) row t, from the staging (not yet overwritten)
        const unsigned char* xs = smem + (isA ? OFF_SK : OFF_SQ);
        const unsigned char* gl = smem + OFF_SL;
        const float xsc = isA ? skf[t] : sqf[t];
#pragma unroll
        for (int k = 0; k < 8; ++k) ps[k] = 0.0f;
        if (t < n) {
          for (int c4 = 0; c4 < TD / 4; ++c4) {
            const float4 xv = staged4_bf16(xs, t, c4);
            const float4 gt = *reinterpret_cast<const float4*>(staged_at(gl, t, 4 * c4, 4u));
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int s2 = sb + k;
              if (s2 <= t) {
                const float4 kv = staged4_bf16(smem + OFF_SK, s2, c4);
                const float4 gs = *reinterpret_cast<const float4*>(staged_at(gl, s2, 4 * c4, 4u));
                float acc = ps[k];
                acc = fmaf(xv.x * kv.x, expf(gt.x - gs.x), acc);
                acc = fmaf(xv.y * kv.y, expf(gt.y - gs.y), acc);
                acc = fmaf(xv.z * kv.z, expf(gt.z - gs.z), acc);
                acc = fmaf(xv.w * kv.w, expf(gt.w - gs.w), acc);
                ps[k] = acc;
              }
            }
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) ps[k] *= xsc * skf[sb + k];
        }
      }
      if (isA) {
        const float bt = bet[t];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int s2 = sb + k;
          A[s2 * TC_ATS + t] = (s2 < t && !plain) ? bt * ps[k] : 0.0f;
        }
      } else {
#pragma unroll
        for (int s4 = 0; s4 < 8; s4 += 4) {
          float pv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) pv[k] = (sb + s4 + k <= t) ? ps[s4 + k] : 0.0f;
          store_split4(smem, OFF_PH, OFF_PL, kmaj_off(t, sb + s4, P_LBO), pv[0], pv[1], pv[2], pv[3]);
        }
      }
    }
    tc::fence_smem_to_async();
    if ((bad = __syncthreads_or(bad) != 0)) break;  // (S2) A and the P tile are complete
    if (warp == ISSUER && !split && nt0 < n_tok) {
      // a chunk without Kbar read q and k in its pair sums: their next copies go now
      copy_q(nt0);
      copy_k(nt0);
    }
    if (!split && nt0 < n_tok) load_beta(nt0, nn);

    if (!wait_warp(&bars[1], it & 1u)) bad = true;
    tc::fence_after_sync();
    if (warp < 4 && !bad) {
      // ---- residuals R = diag(beta) (V - Ktil S0) (v from the staging), substitution, B^T ---
      if (!wait_warp(stv, it & 1u)) bad = true;
      float rr[TC_C];
      {
        float d[16];
        const unsigned char* vs = smem + OFF_SV;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          tc::ld16(tmem + lb + d1 + 16 * h2, d);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int t = 16 * h2 + k;
            const uint16_t vb = t < n ? *reinterpret_cast<const uint16_t*>(staged_at(vs, t, j, 2u)) : uint16_t(0);
            const float vt = __uint_as_float(static_cast<uint32_t>(vb) << 16);
            rr[t] = plain ? bet[t] * vt : bet[t] * (vt - d[k]);
          }
        }
      }
      float* bc = rr;
      if (!plain) {
#pragma unroll
        for (int s2 = 0; s2 < TC_C - 1; ++s2) {
          const float bs = bc[s2];
#pragma unroll
          for (int t4 = (s2 + 1) & ~3; t4 < TC_C; t4 += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(A + s2 * TC_ATS + t4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (t4 + k > s2) bc[t4 + k] = fmaf(-av[k], bs, bc[t4 + k]);
          }
        }
      }
#pragma unroll
      for (int s4 = 0; s4 < TC_C; s4 += 4)
        store_split4(smem, OFF_BH, OFF_BL, kmaj_off(j, s4, T128_LBO), bc[s4], bc[s4 + 1], bc[s4 + 2], bc[s4 + 3]);
    } else if (warp >= 4 && warp < ISSUER) {
      float gv[32];
      if (epi && it > 0) load_gates(prev_t0, prev_n, gv);
      // ---- decay of the state, column c by e^{gamma_C[c]}, before the write accumulates ------
      if (!bad) {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float v[16];
          tc::ld16(tmem + lb + TM_S + 16 * cc, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] *= dC[16 * cc + k];
          tc::st16(tmem + lb + TM_S + 16 * cc, v);
        }
        tc::wait_st();
      }
      // the previous chunk's output, from the other TMEM buffer, while the substitution runs
      // (decided jointly by warps 4-7: the epilogue synchronises them)
      if (!upper_sync_or(bad) && it > 0) store_output(d1 == TM_D1 ? TM_D1B : TM_D1, prev_t0, prev_n, gv);
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    if ((bad = __syncthreads_or(bad) != 0)) break;  // (S3)
    tc::fence_after_sync();

    if (warp == ISSUER) {
      if (nt0 < n_tok) copy_v(nt0);  // the staged v rows are free
      if (epi && (reinterpret_cast<uintptr_t>(p.out_gate) & 15u) == 0u && lane < n) {
        // this chunk's output gates into L2, a chunk before the epilogue reads them
        bulk_prefetch_l2(p.out_gate + ((static_cast<size_t>(b) * T + t0 + lane) * p.H + h) * TD, TD * 4u);
      }
      const uint32_t bh = sbase + OFF_BH, bl = sbase + OFF_BL;
      const uint32_t kh = sbase + OFF_KH, kl = sbase + OFF_KL;
      const uint32_t ph = sbase + OFF_PH, pl = sbase + OFF_PL;
      // state write S^T += B^T Khat and readout O^T = Y^T + B^T P^T (3 x TF32 each)
#pragma unroll 1
      for (int gidx = 0; gidx < 3; ++gidx) {
        const uint32_t a = gidx == 1 ? bl : bh;
        const uint32_t bk = gidx == 2 ? kl : kh, bp = gidx == 2 ? pl : ph;
#pragma unroll
        for (int i = 0; i < TC_C / 8; ++i) {
          const uint64_t ad = tc::smem_desc(a + 2 * i * T128_LBO, T128_LBO, SBO);
          tc::mma_ss(tmem + TM_S, ad, tc::smem_desc(bk + 2 * i * T128_LBO, T128_LBO, SBO), IDESC_P2, 1u);
          tc::mma_ss(tmem + d1 + TC_C, ad, tc::smem_desc(bp + 2 * i * P_LBO, P_LBO, SBO), IDESC_RO, 1u);
        }
      }
      tc::commit(&bars[2]);
    }
    prev_t0 = t0;
    prev_n = n;
    ++it;
    t0 = nt0;
    if (t0 >= n_tok) break;
    n = nn;
    token_stage(n);  // overlaps the MMAs just issued (they read B, Khat and P only)
    nt0 = t0 + TC_C;
    nn = n_tok - nt0 < TC_C ? n_tok - nt0 : TC_C;
    if (split && nt0 < n_tok) {
      copy_q(nt0);
      load_beta(nt0, nn);
    }
  }

  if (!bad) {
    if (!wait_warp(&bars[2], (it - 1) & 1u)) bad = true;
    tc::fence_after_sync();
  }
  bad = __syncthreads_or(bad) != 0;
  if (!bad && warp >= 4 && warp < ISSUER) {
    float gv[32];
    if (epi) load_gates(prev_t0, prev_n, gv);
    store_output((it - 1) & 1u ? TM_D1B : TM_D1, prev_t0, prev_n, gv);
  }
  if (bad) {
    // let every MMA and copy this CTA issued finish (bounded) before the memory is released
    if (warp == ISSUER) {
      tc::commit(&bars[3]);
      if (nq > 0) (void)mbar_wait(stq, (nq - 1u) & 1u);
      if (nk > 0) (void)mbar_wait(stk, (nk - 1u) & 1u);
      if (nv > 0) (void)mbar_wait(stv, (nv - 1u) & 1u);
    }
    (void)mbar_wait(&bars[3], 0u);
    if (tid == 0) atomic_status(p.status, GDN_STATUS_TIMEOUT);
  } else if (warp < ISSUER) {
    // ---- the final state back to the pool row -------------------------------------------
    const int c0 = 64 * (tid >> 7);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float v[16];
      tc::ld16(tmem + lb + TM_S + c0 + 16 * cc, v);
#pragma unroll
      for (int k = 0; k < 16; ++k) Sg[static_cast<size_t>(c0 + 16 * cc + k) * TD + j] = v[k];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, TM_COLS);
}

constexpr int kMaxDevices = 64;

}  // namespace

bool prefill_tc_pk_supported(const DecodeParams& p) {
  // bf16 q, k, v; the decays are fp32; the position coordinate b*T + t is a 32-bit copy coordinate
  return p.D == TD && p.DV == TD && p.dlam == TD && (p.flags & GDN_QKV_BF16) != 0u &&
         (p.flags & GDN_FUSE_CONV) == 0u &&
         static_cast<long long>(p.B) * p.T <= 0x7fffffffLL &&
         (reinterpret_cast<uintptr_t>(p.lam) & 15u) == 0u;  // (the decays' tensor map needs it)
}

cudaError_t launch_prefill_tc_pk(const DecodeParams& p, cudaStream_t stream) {
  static std::atomic<int> configured[kMaxDevices];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    err = cudaFuncSetAttribute(gdn_prefill_tc_pk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(PK_SMEM));
    if (err != cudaSuccess) return err;
    configured[dev].store(1, std::memory_order_relaxed);
  }
  // q, k, v (bf16) and the log decays (fp32) as [B*T][H][128] tensors: boxes of 128 bytes of
  // elements x 1 head x 32 positions
  TokenMapsPK maps;
  const cuuint64_t dims[3] = {TD, static_cast<cuuint64_t>(p.H), static_cast<cuuint64_t>(p.B) * static_cast<cuuint64_t>(p.T)};
  const cuuint64_t s16[2] = {TD * 2u, static_cast<cuuint64_t>(p.H) * TD * 2u};
  const cuuint64_t s32[2] = {TD * 4u, static_cast<cuuint64_t>(p.H) * TD * 4u};
  const cuuint32_t box16[3] = {64u, 1u, static_cast<cuuint32_t>(TC_C)};
  const cuuint32_t box32[3] = {32u, 1u, static_cast<cuuint32_t>(TC_C)};
  const void* bases[3] = {p.q, p.k, p.v};
  CUtensorMap* out[3] = {&maps.q, &maps.k, &maps.v};
  for (int i = 0; i < 3; ++i) {
    err = encode_tiled(out[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, bases[i], dims, s16, box16, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
  }
  err = encode_tiled(&maps.lam, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.lam, dims, s32, box32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.H));
  cfg.blockDim = dim3(TC_NT);
  cfg.dynamicSmemBytes = PK_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, gdn_prefill_tc_pk_kernel, p, maps);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace gdn
