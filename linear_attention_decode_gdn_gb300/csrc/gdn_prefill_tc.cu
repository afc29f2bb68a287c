// gdn_prefill_tc.cu -- chunked prefill on the tcgen05 tensor cores (head size 128, per-head decay).
//
// Evolution article, "Prefill中的Chunk微观并行" (the six-step order of "完整计算顺序"): inside a
// chunk of C = 32 tokens with cumulative log-decays gamma_t,
//   A_ts = beta_t e^{gamma_t - gamma_s} k_t.k_s  (s < t),   P_ts = e^{gamma_t - gamma_s} q_t.k_s  (s <= t)
//   (I + A) B = diag(beta) (V - Ktil S0),  Ktil_t = e^{gamma_t} k_t
//   O_t = e^{gamma_t} (q_t S0) + sum_{s <= t} P_ts B_s
//   S_C = e^{gamma_C} S0 + Khat^T B,          Khat_s = e^{gamma_C - gamma_s} k_s
// i.e. the decode step's recurrence token for token (decay first, residual on the decayed
// state, outer-product write, post-update readout; S[dk][dv], o = S^T q).  The plain update
// (b = beta v) has no A.
//
// The matrix products run on the fifth-generation tensor cores (kind::tf32) with three-term
// TF32 splitting, x = hi + lo with hi = x truncated to TF32 (the tensor core truncates its
// fp32 operands the same way) and X Y ~ Xhi Yhi + Xlo Yhi + Xhi Ylo, which keeps fp32
// accuracy (error ~2^-20 relative per term):
//   pair sums   [K; Q] K^T            (M = 64, N = 32, K = 128)
//   state read  S^T [K; Q]^T          (M = 128, N = 64, K = 128; S from TMEM)
//   state write S^T <- S^T + B^T Khat (M = 128, N = 128, K = 32)
//   readout     O^T <- O^T + B^T P^T  (M = 128, N = 32, K = 32)
// The fp32 state lives in tensor memory for the whole prompt, transposed (TMEM lane j = value
// column, TMEM column c = key channel), with its TF32 remainder lo(S) beside it; shared memory
// holds the operand tiles only.  The forward substitution stays on the CUDA cores
// (column-parallel, one thread per value column).  One CTA of 8 warps per (request, head):
// warps 0-3 own value columns j = tid for the substitution; warps 4-7 (the same TMEM lanes)
// form the pair-sum matrices, rescale the state and store the outputs meanwhile; a ninth warp
// issues the MMAs (one elected lane) and does nothing else, so no compute warp ever waits on
// the tensor core's issue queue.  The next chunk's token stage runs
// while the state-write and readout MMAs of the current chunk execute.
//
// With the fused conv (evolution article, "去掉分母引入卷积") the token stage stages bf16 mixed_qkv
// rows with a three-position halo and runs the width-4 conv + SiLU there (taps and biases in
// shared memory, the slot's conv state standing in for the positions before the prompt); the
// conv outputs are fp32 and take the three-term split like fp32 inputs.
#include <atomic>

#include "gdn_tc.cuh"
#include "gdn_tmap.h"

namespace gdn {
namespace {

constexpr int TD = 128;      // head size of this kernel
constexpr int TC_C = 32;     // tokens per chunk
constexpr int TC_NT = 288;   // threads per CTA: 8 compute warps and the MMA-issuing warp
constexpr int ISSUER = 8;    // the warp that issues every MMA and does nothing else
constexpr int TC_ATS = TC_C + 4;

// Operand tiles (K-major, no swizzle; element (r, k) at (r/8)*128 + (k/4)*LBO + (r%8)*16 + (k%4)*4,
// so groups of 8 rows are adjacent and the k direction steps by LBO = rows/8 * 128 bytes).
constexpr uint32_t X_LBO = (2 * TC_C / 8) * 128;   // [K; Q] rows: 64 x 128      (1024)
constexpr uint32_t T128_LBO = (TD / 8) * 128;      // Khat^T, B^T:  128 x 32     (2048)
constexpr uint32_t P_LBO = (TC_C / 8) * 128;       // P:            32 x 32      (512)
constexpr uint32_t SBO = 128;

// Staging of the raw token inputs, one chunk ahead: per tensor (q, k, v) the chunk's 32 rows
// of 128 elements as 128-byte column boxes ([box][row][128 bytes]: 2 boxes for bf16, 4 for
// fp32), each written by one 3-D TMA copy with the 128-byte swizzle (16-byte chunk c of row t
// at chunk position c ^ (t % 8)), so that both the row-wise token stage and the copies see no
// bank conflicts.
constexpr uint32_t ST_BOX = TC_C * 128;  // bytes of one box

// shared-memory layout (bytes)
constexpr uint32_t OFF_XH = 0;                      // [K; Q] hi  64 x 128
constexpr uint32_t OFF_XL = OFF_XH + 2 * TC_C * TD * 4;
constexpr uint32_t OFF_KH = OFF_XL + 2 * TC_C * TD * 4;  // Khat^T hi 128 x 32
constexpr uint32_t OFF_KL = OFF_KH + TD * TC_C * 4;
constexpr uint32_t OFF_BH = OFF_KL + TD * TC_C * 4;      // B^T hi 128 x 32
constexpr uint32_t OFF_BL = OFF_BH + TD * TC_C * 4;
constexpr uint32_t OFF_PH = OFF_BL + TD * TC_C * 4;      // P hi 32 x 32
constexpr uint32_t OFF_PL = OFF_PH + TC_C * TC_C * 4;
constexpr uint32_t OFF_V = OFF_PL + TC_C * TC_C * 4;     // V row-major 32 x 128 fp32
constexpr uint32_t OFF_A = OFF_V + TC_C * TD * 4;        // A column-major [s][TC_ATS]
constexpr uint32_t OFF_ST = (OFF_A + TC_C * TC_ATS * 4 + 1023u) & ~1023u;  // staging (1024-aligned: swizzle atoms)
constexpr uint32_t OFF_G = OFF_ST + 3 * TC_C * TD * 4;   // gamma, beta, e^gamma, e^{gamma_C - gamma},
                                                         // key and query scale factors, e^-gamma, flags
// Fused conv (GDN_FUSE_CONV, bf16 mixed_qkv; evolution article, "去掉分母引入卷积"): every staged
// box holds the chunk's rows with the three positions before them (35 rows, position t0 - 3 + r
// in row r), padded to whole 1024-byte swizzle atoms (in the first chunk the slot's conv state
// replaces rows 0-2); the head's conv taps and biases sit in the rest of the staging area.
constexpr int CV_ROWS = TC_C + 3;
constexpr uint32_t CV_BOX = 5 * 1024;
constexpr uint32_t CV_CH = 3 * TD;                         // the head's q, k and v channels
constexpr uint32_t OFF_CW = OFF_ST + 3 * 2 * CV_BOX;       // taps of channel c as one float4
constexpr uint32_t OFF_CB = OFF_CW + CV_CH * 16;           // biases
static_assert(CV_ROWS * 128 <= CV_BOX && OFF_CB + CV_CH * 4 <= OFF_G, "fused-conv staging");
constexpr uint32_t OFF_BAR = OFF_G + 8 * TC_C * 4;       // mbarriers: ps, p1, p2, drain, then one
                                                         // per compute warp for its staged rows
constexpr uint32_t OFF_TMEM = OFF_BAR + 12 * 8;
constexpr uint32_t TC_SMEM = OFF_TMEM + 16;

// TMEM columns
constexpr uint32_t TM_S = 0;     // S^T fp32, 128 columns
constexpr uint32_t TM_L = 128;   // lo(S^T)
constexpr uint32_t TM_D1 = 256;  // [K S | Q S] -> [. | O], 64 columns, two buffers (chunk parity)
constexpr uint32_t TM_PS = 320;  // pair sums (M = 64 layout), 32 columns
constexpr uint32_t TM_D1B = 352;
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t IDESC_PS = tc::idesc_tf32(64, 32);
constexpr uint32_t IDESC_P1 = tc::idesc_tf32(128, 64);
constexpr uint32_t IDESC_P2 = tc::idesc_tf32(128, 128);
constexpr uint32_t IDESC_RO = tc::idesc_tf32(128, 32);

__device__ __forceinline__ uint32_t kmaj_off(int r, int k, uint32_t lbo) {
  return static_cast<uint32_t>((r >> 3) * SBO + (k >> 2) * lbo + (r & 7) * 16 + (k & 3) * 4);
}

// hi / lo of four values, stored as two float4 at byte offset `off` of the hi and lo tiles
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

// Elements 4g .. 4g+3 of row t of staged tensor `tensor` (0 q, 1 k, 2 v; bf16 or fp32), as
// float: the 128-byte box that holds them, then the swizzled 16-byte chunk.
__device__ __forceinline__ float4 staged4(const unsigned char* st, int tensor, int t, int g, bool bf16) {
  const uint32_t esz = bf16 ? 2u : 4u;
  const uint32_t byte = 4u * static_cast<uint32_t>(g) * esz;
  const uint32_t inb = byte & 127u;
  const unsigned char* at = st + static_cast<uint32_t>(tensor) * (TC_C * TD * esz) + (byte >> 7) * ST_BOX +
                            static_cast<uint32_t>(t) * 128u +
                            ((((inb >> 4) ^ (static_cast<uint32_t>(t) & 7u)) << 4) | (inb & 15u));
  if (bf16) {
    const uint2 u = *reinterpret_cast<const uint2*>(at);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
  }
  return *reinterpret_cast<const float4*>(at);
}

// Fused conv: byte offset of bf16 element c of tensor `tensor` at staged row r
__device__ __forceinline__ uint32_t conv_at(int tensor, int r, int c) {
  const uint32_t byte = 2u * static_cast<uint32_t>(c);
  const uint32_t inb = byte & 127u;
  return OFF_ST + static_cast<uint32_t>(tensor) * (2 * CV_BOX) + (byte >> 7) * CV_BOX + static_cast<uint32_t>(r) * 128u +
         ((((inb >> 4) ^ (static_cast<uint32_t>(r) & 7u)) << 4) | (inb & 15u));
}

// Fused conv: pre-conv inputs, channels 4g .. 4g+3 of tensor `tensor`, at staged row r (position
// t0 - 3 + r).
__device__ __forceinline__ float4 conv_in4(const unsigned char* smem, int tensor, int r, int g) {
  const uint32_t byte = 8u * static_cast<uint32_t>(g);
  const uint32_t inb = byte & 127u;
  const unsigned char* at = smem + OFF_ST + static_cast<uint32_t>(tensor) * (2 * CV_BOX) + (byte >> 7) * CV_BOX +
                            static_cast<uint32_t>(r) * 128u +
                            ((((inb >> 4) ^ (static_cast<uint32_t>(r) & 7u)) << 4) | (inb & 15u));
  const uint2 u = *reinterpret_cast<const uint2*>(at);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xffff0000u));
}

// Width-4 causal conv + SiLU of one channel from its inputs at positions t-3 .. t (tap 3 on the
// current one), in the decode kernels' product order (a missing bias is staged as 0); the SiLU
// through the fast intrinsics (relative error a few parts in 10^7; z e^-z -> 0 below -88).
__device__ __forceinline__ float conv1(float x0, float x1, float x2, float x3, float4 w, float bias) {
  float acc = x0 * w.x;
  acc = fmaf(x1, w.y, acc);
  acc = fmaf(x2, w.z, acc);
  acc = fmaf(x3, w.w, acc);
  const float z = acc + bias;
  return z * __fdividef(1.0f, 1.0f + __expf(-z));
}

// The taps (one float4 per channel) and biases of channels 4g .. 4g+3 of tensor `tensor`.
struct ConvW4 {
  float4 w0, w1, w2, w3, cb;
};
__device__ __forceinline__ ConvW4 conv_w4(const unsigned char* smem, int tensor, int g) {
  const float4* w = reinterpret_cast<const float4*>(smem + OFF_CW) + tensor * TD + 4 * g;
  return {w[0], w[1], w[2], w[3], *(reinterpret_cast<const float4*>(smem + OFF_CB) + tensor * (TD / 4) + g)};
}

// Four channels of the conv output from their input rows at positions t-3 .. t.
__device__ __forceinline__ float4 conv4(const ConvW4& w, float4 a, float4 b, float4 c, float4 d) {
  return make_float4(conv1(a.x, b.x, c.x, d.x, w.w0, w.cb.x), conv1(a.y, b.y, c.y, d.y, w.w1, w.cb.y),
                     conv1(a.z, b.z, c.z, d.z, w.w2, w.cb.z), conv1(a.w, b.w, c.w, d.w, w.w3, w.cb.w));
}

// The token tensors q, k, v as 3-D tensor maps (element, head, position over all requests):
// dims {128, H, B*T}, boxes {128 bytes of elements, 1, 32}, 128-byte swizzle.
struct TokenMaps {
  CUtensorMap q, k, v;
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

// Bounded wait for phase `parity` of `bar`, the same answer in every lane of the warp (the
// TMEM loads and stores that follow are warp-collective).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// CONV: q, k, v are the width-4 conv + SiLU of bf16 mixed_qkv rows (the maps cover its q, k and
// v thirds), through the slot's conv state, which afterwards holds the prompt's last three inputs.
template <bool CONV>
__global__ void __launch_bounds__(TC_NT, 1) gdn_prefill_tc_kernel(const DecodeParams p, const __grid_constant__ TokenMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / p.H;
  const int h = blockIdx.x - b * p.H;
  const uint32_t fl = p.flags;
  const bool bf16 = (fl & GDN_QKV_BF16) != 0u;
  const bool plain = (fl & GDN_PLAIN_UPDATE) != 0u;
  const bool l2 = (fl & GDN_NO_QK_L2NORM) == 0u;
  // bf16 inputs are exact TF32 values: the products run on the raw q and k (one TF32 term
  // for the pair sums, two for the state read) and the L2-norm scales are applied to the
  // results; fp32 inputs (and conv outputs) are split into hi and lo after normalisation
  const bool exact = bf16 && !CONV;
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

  float* gam = reinterpret_cast<float*>(smem + OFF_G);
  float* bet = gam + TC_C;
  float* eg = gam + 2 * TC_C;
  float* ek = gam + 3 * TC_C;
  float* skf = gam + 4 * TC_C;  // per-token key scale applied to the products (1 when normalised in place)
  float* sqf = gam + 5 * TC_C;  // per-token query scale
  float* ein = gam + 6 * TC_C;  // e^{-gamma}
  int* ratio_split = reinterpret_cast<int*>(gam + 7 * TC_C);  // e^{gamma_t - gamma_s} as e^gamma_t e^-gamma_s
  float* V = reinterpret_cast<float*>(smem + OFF_V);
  float* A = reinterpret_cast<float*>(smem + OFF_A);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* stbar = bars + 4;  // the staging copies of a chunk
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
  const uint32_t esz = bf16 ? 2u : 4u;
  const int wq = warp & 3;

  bool bad = false;
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1u);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- raw token rows of the chunk at t0 into the staging boxes (3-D TMA) --------------------
  // The MMA-issuing warp copies the chunk's q, k and v rows as 128-byte column boxes of the
  // token tensor maps (one copy per box, all counted on one mbarrier); it is idle while the
  // compute warps run the token stage, so the copies cost the chunk's critical path nothing.
  // (Per-row bulk copies, and per-lane 16-byte cp.async, each held the compute warps about
  // 2.5 K cycles a chunk.)  Warp 4 loads the chunk's gates into registers (lane = token).
  uint32_t st_par = 0;     // (compute warps) phase of the staging barrier the next token stage waits for
  uint32_t st_loads = 0;   // (issuer) staging loads issued; the last one completes phase (st_loads - 1) & 1
  float pf_lam = 0.0f, pf_beta = 0.0f;
  const int nbox = bf16 ? 2 : 4;
  auto prefetch = [&](int t0, int n) {
    if (warp == ISSUER) {
      if (CONV) {
        // 35 rows from position t0 - 3 (before the request's first row the copy reads the
        // previous request's rows or, at coordinate -3, the fill value: the conv state stands in)
        tc::expect_tx(stbar, 3u * 2u * CV_ROWS * 128u);
        const int z = b * T + t0 - 3;
#pragma unroll
        for (int tensor = 0; tensor < 3; ++tensor) {
          const CUtensorMap* map = tensor == 0 ? &maps.q : (tensor == 1 ? &maps.k : &maps.v);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_3d(smem_addr(smem + OFF_ST + static_cast<uint32_t>(tensor) * (2 * CV_BOX) + bx * CV_BOX), map,
                        bx * 64, h, z, stbar);
        }
      } else {
        tc::expect_tx(stbar, 3u * static_cast<uint32_t>(nbox) * ST_BOX);
        const int z = b * T + t0;
#pragma unroll
        for (int tensor = 0; tensor < 3; ++tensor) {
          const CUtensorMap* map = tensor == 0 ? &maps.q : (tensor == 1 ? &maps.k : &maps.v);
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_3d(smem_addr(smem + OFF_ST + static_cast<uint32_t>(tensor) * (TC_C * TD * esz) + bx * ST_BOX),
                        map, bx * static_cast<int>(128u / esz), h, z, stbar);
        }
      }
      ++st_loads;
    }
    if (warp == 4) {
      const size_t gi = (static_cast<size_t>(b) * T + t0 + lane) * p.H + h;
      pf_lam = lane < n ? __ldg(p.lam + gi) : 0.0f;
      pf_beta = lane < n ? (p.beta ? __ldg(p.beta + gi) : 1.0f) : 0.0f;
    }
  };
  prefetch(0, n_tok < TC_C ? n_tok : TC_C);

  if (CONV && warp < ISSUER) {
    // the head's conv taps and biases for the compute warps (visible after the barrier that
    // follows the TMEM allocation)
    for (int i = tid; i < static_cast<int>(CV_CH); i += ISSUER * 32) {
      const int ch = (i >> 7) * p.H * TD + h * TD + (i & (TD - 1));
      reinterpret_cast<float4*>(smem + OFF_CW)[i] = __ldg(reinterpret_cast<const float4*>(p.conv_w) + ch);
      reinterpret_cast<float*>(smem + OFF_CB)[i] = p.conv_b != nullptr ? __ldg(p.conv_b + ch) : 0.0f;
    }
  }

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
    const int c0 = 64 * (tid >> 7);  // warps 0-3 columns 0..63, warps 4-7 columns 64..127
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


  // ---- token stage (from the staging rows): [K; Q] tiles, V, gates, norm scales -------------
  // warps 0-3: key rows t = 8 w + (lane & 7), channel groups g = (lane >> 3) + 4 i (4 channels
  // each), then the value rows 8w..8w+7; warps 4-7: query rows the same way; warp 4 also the
  // gates.
  // Ends with the pair-sum MMAs of the chunk issued (they need nothing of the state).
  int t0 = 0;  // the chunk's first position
  auto token_stage = [&](int n) {
   if (warp < ISSUER) {
    if (!wait_warp(stbar, st_par)) bad = true;  // the chunk's rows have landed
    st_par ^= 1u;
    const int t = 8 * wq + (lane & 7);
    const int g0 = lane >> 3;
    const bool live = t < n;
    const bool isk = warp < 4;
    const unsigned char* st = smem + OFF_ST;
    const int r = isk ? t : TC_C + t;
    float4 x[8];
    float ss = 0.0f;
    if (CONV) {
      // the conv outputs of the warp's eight rows, first with lane = channel group over a
      // sliding window of staged rows (row u's output from staged rows u .. u+3, positions
      // u-3 .. u; taps and biases loaded once), parked in a per-warp scratch in the [K; Q]
      // remainder tile (free until the split below: row u at 512 u, channel group g in 16-byte
      // slot g ^ u, conflict-free both ways), then read back with this thread's row and groups
      const int tensor = isk ? 1 : 0;
      const int r0 = 8 * wq;
      unsigned char* scr = smem + OFF_XL + warp * 4096;
      {
        const ConvW4 cw = conv_w4(smem, tensor, lane);
        float4 xa = conv_in4(smem, tensor, r0, lane), xb = conv_in4(smem, tensor, r0 + 1, lane),
               xc = conv_in4(smem, tensor, r0 + 2, lane);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 xd = conv_in4(smem, tensor, r0 + u + 3, lane);
          *reinterpret_cast<float4*>(scr + u * 512 + ((lane ^ u) << 4)) =
              r0 + u < n ? conv4(cw, xa, xb, xc, xd) : make_float4(0.f, 0.f, 0.f, 0.f);
          xa = xb;
          xb = xc;
          xc = xd;
        }
      }
      __syncwarp();
      const int tl = lane & 7;
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = *reinterpret_cast<const float4*>(scr + tl * 512 + (((g0 + 4 * i) ^ tl) << 4));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[i] = live ? staged4(st, isk ? 1 : 0, t, g0 + 4 * i, bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += x[i].x * x[i].x + x[i].y * x[i].y + x[i].z * x[i].z + x[i].w * x[i].w;
    if (warp == 4) {  // gates of the chunk, lane = token
      const bool lv = lane < n;
      float lam = pf_lam, be = pf_beta;
      if ((fl & GDN_GATE_RAW) && lv) {
        lam = log_sigmoidf_(lam);
        if (p.beta) be = sigmoidf_(be);
      }
      float g = lam;  // inclusive prefix sum over the chunk
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, g, off);
        if (lane >= off) g += y;
      }
      const float gC = __shfl_sync(0xffffffffu, g, TC_C - 1);
      gam[lane] = g;
      bet[lane] = be;
      eg[lane] = expf(g);
      ek[lane] = expf(gC - g);
      // the ratio e^{gamma_t - gamma_s} (s <= t) splits into two exponentials while e^-gamma
      // stays finite (the chunk's total log-decay above -80); else it is formed per pair
      const bool split = gC >= -80.0f;
      ein[lane] = split ? expf(-g) : 0.0f;
      if (lane == 0) *ratio_split = split ? 1 : 0;
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 8);
    ss += __shfl_xor_sync(0xffffffffu, ss, 16);
    const float sc = (l2 ? rsqrtf(ss + p.l2_eps) : 1.0f) * (isk ? 1.0f : p.q_scale);
    if ((lane >> 3) == 0) (isk ? skf : sqf)[t] = exact ? sc : 1.0f;
    if (CONV) asm volatile("bar.sync 1, 256;" ::: "memory");  // every warp's scratch is read
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = g0 + 4 * i;
      const float a0 = x[i].x * sc, a1 = x[i].y * sc, a2 = x[i].z * sc, a3 = x[i].w * sc;
      if (exact)  // the raw values: exact TF32, no remainder
        *reinterpret_cast<float4*>(smem + OFF_XH + kmaj_off(r, 4 * g, X_LBO)) = x[i];
      else
        store_split4(smem, OFF_XH, OFF_XL, kmaj_off(r, 4 * g, X_LBO), a0, a1, a2, a3);
    }
    if (CONV) {
      // value rows v0 .. v0+3 (four per compute warp), channels 4 lane .. 4 lane + 3: a sliding
      // window of input rows
      const int v0 = 16 * (warp >> 2) + 4 * wq;
      const ConvW4 cw = conv_w4(smem, 2, lane);
      float4 xa = conv_in4(smem, 2, v0, lane), xb = conv_in4(smem, 2, v0 + 1, lane), xc = conv_in4(smem, 2, v0 + 2, lane);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int tv = v0 + u;
        const float4 xd = conv_in4(smem, 2, tv + 3, lane);
        reinterpret_cast<float4*>(V + tv * TD)[lane] =
            tv < n ? conv4(cw, xa, xb, xc, xd) : make_float4(0.f, 0.f, 0.f, 0.f);
        xa = xb;
        xb = xc;
        xc = xd;
      }
    } else if (isk) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int tv = 8 * wq + u;
        reinterpret_cast<float4*>(V + tv * TD)[lane] =
            tv < n ? staged4(st, 2, tv, lane, bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
   }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();  // gates, scales, tiles visible; the staging rows are free again
    tc::fence_after_sync();
    if (warp == ISSUER) {
      // pair sums [K; Q] K^T  (exact inputs: one TF32 term; else hi hi, lo hi, hi lo)
      const uint32_t xh = sbase + OFF_XH, xl = sbase + OFF_XL;
      const int ng = exact ? 1 : 3;
#pragma unroll 1
      for (int gidx = 0; gidx < ng; ++gidx) {
        const uint32_t a = gidx == 1 ? xl : xh, bb = gidx == 2 ? xl : xh;
#pragma unroll
        for (int i = 0; i < TD / 8; ++i)
          tc::mma_ss(tmem + TM_PS, tc::smem_desc(a + 2 * i * X_LBO, X_LBO, SBO),
                     tc::smem_desc(bb + 2 * i * X_LBO, X_LBO, SBO), IDESC_PS, (gidx | i) != 0);
      }
      tc::commit(&bars[0]);
    }
  };

  int n = n_tok < TC_C ? n_tok : TC_C;
  if (CONV && warp < ISSUER) {
    // first chunk: the slot's conv state (pre-conv inputs at positions -3 .. -1) over staged
    // rows 0-2, once the copy has landed there (the token stage's wait then finds it complete)
    if (!wait_warp(stbar, 0u)) bad = true;
    const uint16_t* cp = static_cast<const uint16_t*>(p.conv_pool);
    for (int i = tid; i < static_cast<int>(CV_CH); i += ISSUER * 32) {
      const int tensor = i >> 7, c = i & (TD - 1);
      const uint16_t* cs = cp + (static_cast<size_t>(slot) * p.channels + tensor * p.H * TD + h * TD + c) * 3;
#pragma unroll
      for (int r = 0; r < 3; ++r) *reinterpret_cast<uint16_t*>(smem + conv_at(tensor, r, c)) = cs[r];
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the compute warps
  }
  token_stage(n);
  if (TC_C < n_tok) prefetch(TC_C, n_tok - TC_C < TC_C ? n_tok - TC_C : TC_C);
  int prev_t0 = 0, prev_n = 0;
  uint32_t it = 0;

  // readout of a finished chunk from its TMEM output buffer (warps 4-7): lane j of warp 4 + w
  // holds O^T[32 w + j][t]; for each position t < cn the warp stores its 32 columns of the
  // output row (128 contiguous bytes).  (One TMA bulk store per row cost about 2 K cycles a
  // chunk in issue.)
  auto store_output = [&](uint32_t d1, int ct0, int cn) {
    float* orow = p.o + ((static_cast<size_t>(b) * T + ct0) * p.H + h) * TD + j;
    const size_t tstride = static_cast<size_t>(p.H) * TD;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float o[16];
      tc::ld16(tmem + lb + d1 + TC_C + 16 * h2, o);
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (16 * h2 + k < cn) orow[(16 * h2 + k) * tstride] = o[k];
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
      // Khat^T tile (row c, column s): k_s[c] e^{gamma_C - gamma_s}, the normalised key read
      // back from the [K; Q] tile this thread wrote in the token stage (the raw key times its
      // scale for exact inputs, else hi + lo: the same values, kept out of registers across
      // the chunk)
      const int s = 8 * warp + (lane & 7);
      const float f = ek[s], sk = skf[s];
      const int g0 = lane >> 3;
#pragma unroll(CONV ? 2 : 8)
      for (int i = 0; i < 8; ++i) {
        const int c = 4 * (g0 + 4 * i);
        const uint32_t xo = kmaj_off(s, c, X_LBO);
        float4 a = *reinterpret_cast<const float4*>(smem + OFF_XH + xo);
        if (exact) {
          a.x *= sk;
          a.y *= sk;
          a.z *= sk;
          a.w *= sk;
        } else {
          const float4 l = *reinterpret_cast<const float4*>(smem + OFF_XL + xo);
          a.x += l.x;
          a.y += l.y;
          a.z += l.z;
          a.w += l.w;
        }
        store_split1(smem, OFF_KH, OFF_KL, kmaj_off(c + 0, s, T128_LBO), a.x * f);
        store_split1(smem, OFF_KH, OFF_KL, kmaj_off(c + 1, s, T128_LBO), a.y * f);
        store_split1(smem, OFF_KH, OFF_KL, kmaj_off(c + 2, s, T128_LBO), a.z * f);
        store_split1(smem, OFF_KH, OFF_KL, kmaj_off(c + 3, s, T128_LBO), a.w * f);
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    if ((bad = __syncthreads_or(bad) != 0)) break;  // (S1)
    tc::fence_after_sync();

    if (warp == ISSUER) {  // the whole warp: one elected lane issues
      // state read S^T [K; Q]^T  (A = S from TMEM: its fp32 bits read as TF32 are hi(S)):
      // hi(S) X, lo(S) X (and hi(S) lo(X) for inexact inputs)
      const uint32_t xh = sbase + OFF_XH, xl = sbase + OFF_XL;
#pragma unroll 1
      for (int gidx = 0; gidx < 3; ++gidx) {
        if (exact && gidx == 1) continue;
        const uint32_t a = tmem + (gidx == 2 ? TM_L : TM_S), bb = gidx == 1 ? xl : xh;
#pragma unroll
        for (int i = 0; i < TD / 8; ++i)
          tc::mma_ts(tmem + d1, a + 8 * i, tc::smem_desc(bb + 2 * i * X_LBO, X_LBO, SBO), IDESC_P1,
                     (gidx | i) != 0);
      }
      tc::commit(&bars[1]);
    } else {
      // ---- A (strictly lower, times beta) and P (lower with the diagonal) from the pair sums
      // (issued at the end of the token stage), while the state read runs, on all eight compute
      // warps. M = 64 accumulator: row m sits in lane 32 (m / 16) + m % 16, so warps w and w + 4
      // (the same lane quarter) hold the k.k rows t = 16 (w % 2) + lane for w % 4 < 2 and the q.k
      // rows for w % 4 >= 2 (lanes < 16). Warp group G = w / 4 takes the source tokens
      // s = 16 G .. 16 G + 15: lanes < 16 the first eight, lanes >= 16 the last eight of their
      // row (shuffled from lane - 16).
      if (!wait_warp(&bars[0], it & 1u)) bad = true;
      tc::fence_after_sync();
      const int G = warp >> 2, half = lane >> 4;
      float a16[16], ps[8];
      tc::ld16(tmem + lb + TM_PS + 16 * G, a16);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float up = __shfl_sync(0xffffffffu, a16[8 + k], lane & 15);
        ps[k] = half ? up : a16[k];
      }
      const bool split = *ratio_split != 0;
      const int t = 16 * (warp & 1) + (lane & 15);
      const int sb = 16 * G + 8 * half;  // this thread's first source token
      const float egt = eg[t], gt = gam[t];
      if ((warp & 2) == 0) {
        const float bt = bet[t] * skf[t];
        if (split) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int s2 = sb + k;
            A[s2 * TC_ATS + t] = (s2 < t && !plain) ? bt * (ps[k] * skf[s2]) * (egt * ein[s2]) : 0.0f;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int s2 = sb + k;
            A[s2 * TC_ATS + t] = (s2 < t && !plain) ? bt * (ps[k] * skf[s2]) * expf(gt - gam[s2]) : 0.0f;
          }
        }
      } else {
        const float qt = sqf[t];
#pragma unroll
        for (int s4 = 0; s4 < 8; s4 += 4) {
          float pv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int s2 = sb + s4 + k;
            const float rr = split ? egt * ein[s2] : expf(gt - gam[s2]);
            pv[k] = s2 <= t ? qt * (ps[s4 + k] * skf[s2]) * rr : 0.0f;
          }
          store_split4(smem, OFF_PH, OFF_PL, kmaj_off(t, sb + s4, P_LBO), pv[0], pv[1], pv[2], pv[3]);
        }
      }
    }
    tc::fence_smem_to_async();
    if ((bad = __syncthreads_or(bad) != 0)) break;  // (S2) A and the P tile are complete

    if (!wait_warp(&bars[1], it & 1u)) bad = true;
    tc::fence_after_sync();
    {
      if (warp < 4 && !bad) {
        // ---- residuals R, forward substitution, the B^T tile -------------------------------
        float rr[TC_C];
        {
          float d[16];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            tc::ld16(tmem + lb + d1 + 16 * h2, d);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int t = 16 * h2 + k;
              const float vt = V[t * TD + j];
              rr[t] = plain ? bet[t] * vt : bet[t] * (vt - (eg[t] * skf[t]) * d[k]);
            }
          }
          // Y = e^{gamma_t} (q_t S0), in place: the readout MMA accumulates P B onto it
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            tc::ld16(tmem + lb + d1 + TC_C + 16 * h2, d);
#pragma unroll
            for (int k = 0; k < 16; ++k) d[k] *= eg[16 * h2 + k] * sqf[16 * h2 + k];
            tc::st16(tmem + lb + d1 + TC_C + 16 * h2, d);
          }
        }
        // forward substitution (I + A) B = R, right-looking: once row s is final it is folded
        // into every later row
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
        tc::wait_st();
      } else if (warp >= 4 && warp < ISSUER) {
        // ---- decay of the state by e^{gamma_C} before the write accumulates onto it ---------
        if (!bad) {
          const float dC = eg[TC_C - 1];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            float v[16];
            tc::ld16(tmem + lb + TM_S + 16 * cc, v);
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] *= dC;
            tc::st16(tmem + lb + TM_S + 16 * cc, v);
          }
          tc::wait_st();
        }
        // the previous chunk's output, from the other TMEM buffer, while the substitution runs
        if (!bad && it > 0) store_output(d1 == TM_D1 ? TM_D1B : TM_D1, prev_t0, prev_n);
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    if ((bad = __syncthreads_or(bad) != 0)) break;  // (S3)
    tc::fence_after_sync();

    if (warp == ISSUER) {
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
    t0 += TC_C;
    if (t0 >= n_tok) break;
    n = n_tok - t0 < TC_C ? n_tok - t0 : TC_C;
    token_stage(n);  // overlaps the MMAs just issued (they read B, Khat and P only)
    if (t0 + TC_C < n_tok) prefetch(t0 + TC_C, n_tok - t0 - TC_C < TC_C ? n_tok - t0 - TC_C : TC_C);
  }

  if (!bad) {
    if (!wait_warp(&bars[2], (it - 1) & 1u)) bad = true;
    tc::fence_after_sync();
  }
  bad = __syncthreads_or(bad) != 0;
  if (!bad && warp >= 4 && warp < ISSUER) store_output((it - 1) & 1u ? TM_D1B : TM_D1, prev_t0, prev_n);
  if (bad) {
    // let every MMA this CTA issued finish (bounded) before the tensor memory is released
    if (warp == ISSUER) tc::commit(&bars[3]);
    (void)mbar_wait(&bars[3], 0u);
    if (warp == ISSUER && st_loads > 0) (void)mbar_wait(stbar, (st_loads - 1u) & 1u);  // staging copies in flight
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
    if (CONV) {
      // the conv state keeps the last three inputs of (old state, prompt), bit-exact; each
      // thread reads all three of a channel's before it writes them
      uint16_t* cp = static_cast<uint16_t*>(p.conv_pool);
      const uint16_t* mx = static_cast<const uint16_t*>(p.mixed);
      for (int i = tid; i < static_cast<int>(CV_CH); i += ISSUER * 32) {
        const int ch = (i >> 7) * p.H * TD + h * TD + (i & (TD - 1));
        uint16_t* cs = cp + (static_cast<size_t>(slot) * p.channels + ch) * 3;
        uint16_t nb[3];
#pragma unroll
        for (int col = 0; col < 3; ++col) {
          const int pos = n_tok - 3 + col;
          nb[col] = pos >= 0 ? __ldg(mx + (static_cast<size_t>(b) * T + pos) * p.channels + ch) : cs[pos + 3];
        }
#pragma unroll
        for (int col = 0; col < 3; ++col) cs[col] = nb[col];
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, TM_COLS);
}

constexpr int kMaxDevices = 64;

}  // namespace

bool prefill_tc_supported(const DecodeParams& p) {
  // (the token tensors' position coordinate b*T + t is a 32-bit tensor-copy coordinate; the
  // fused conv stages bf16 mixed_qkv rows only)
  const bool conv = (p.flags & GDN_FUSE_CONV) != 0u;
  return p.D == TD && p.dlam == 1 && (p.flags & (GDN_GATE_KDA | GDN_OUT_NORM_GATE)) == 0u &&
         (!conv || (p.flags & GDN_QKV_BF16) != 0u) && static_cast<long long>(p.B) * p.T <= 0x7fffffffLL;
}

namespace {

template <bool CONV>
cudaError_t launch_prefill_tc_k(const DecodeParams& p, cudaStream_t stream) {
  static std::atomic<int> configured[kMaxDevices];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    err = cudaFuncSetAttribute(gdn_prefill_tc_kernel<CONV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(TC_SMEM));
    if (err != cudaSuccess) return err;
    configured[dev].store(1, std::memory_order_relaxed);
  }
  // q, k, v as [B*T][H][128] tensors: boxes of 128 bytes of elements x 1 head x 32 positions
  // (fused conv: the q, k and v thirds of the [B*T][3*H*128] mixed_qkv rows, 35 positions)
  TokenMaps maps;
  const bool bf16 = (p.flags & GDN_QKV_BF16) != 0u;
  const cuuint64_t esz = bf16 ? 2u : 4u;
  const cuuint64_t row = CONV ? static_cast<cuuint64_t>(p.channels) : static_cast<cuuint64_t>(p.H) * TD;
  const cuuint64_t dims[3] = {TD, static_cast<cuuint64_t>(p.H), static_cast<cuuint64_t>(p.B) * static_cast<cuuint64_t>(p.T)};
  const cuuint64_t strides[2] = {TD * esz, row * esz};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128u / esz), 1u, static_cast<cuuint32_t>(CONV ? CV_ROWS : TC_C)};
  const CUtensorMapDataType ty = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const size_t third = static_cast<size_t>(p.H) * TD * esz;
  const void* bases[3] = {p.q, p.k, p.v};
  if (CONV)
    for (int i = 0; i < 3; ++i) bases[i] = static_cast<const unsigned char*>(p.mixed) + i * third;
  CUtensorMap* out[3] = {&maps.q, &maps.k, &maps.v};
  for (int i = 0; i < 3; ++i) {
    err = encode_tiled(out[i], ty, 3, bases[i], dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.H));
  cfg.blockDim = dim3(TC_NT);
  cfg.dynamicSmemBytes = TC_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, gdn_prefill_tc_kernel<CONV>, p, maps);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const DecodeParams& p, cudaStream_t stream) {
  return (p.flags & GDN_FUSE_CONV) ? launch_prefill_tc_k<true>(p, stream) : launch_prefill_tc_k<false>(p, stream);
}

}  // namespace gdn
