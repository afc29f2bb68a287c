// gdn_decode.cu -- the decode-step kernels (dense, DeltaLog append, merge, auto step) for
// square heads handled by one CTA each (dk == dv in {16, 32, 64, 128}), and the shape dispatch
// of every decode launch. gdn_decode_x.cu (kernel in gdn_decode_kernel.cuh) builds the other
// shapes: dk != dv, and heads split along dv over two CTAs. That kernel computes the same step
// for these shapes too, but measured about 2.5% slower on the append of square heads (a short,
// latency-bound CTA: the compiler schedules the general form differently), so the square
// one-CTA path keeps this kernel.
//
// One CTA owns one (request, head): it is the single writer of that head's
// state / base tile, its output row and its log entries (DeltaLog notes,
// Sec. 2.6 / Fig. 5 split the tile along dv across CTAs and need a separate
// finalize pass for the shared metadata; on GB300 a whole 128x128 fp32 tile
// (64 KiB) fits in shared memory three times per SM, so the head is not split
// and the metadata commit needs no second pass).
//
// Per CTA (8 compute warps + 1 copy-issuing warp):
//   launch    programmatic stream serialisation: the CTA lets the next launch schedule at
//             once and waits for the previous grid before its first read (first-wave
//             CTAs prefetch their tile into L2 before that wait).
//   prologue  the copy warp starts the TMA bulk copies of the tile (4 row chunks for
//             dk = 128) and the log copy (append: the first L entries once L is read;
//             merge: all C); the compute warps load the gates and q/k/v (or run the
//             width-4 conv + SiLU) and form the decays exp(ell').  One barrier.
//   replay    while the tile is in flight, one warp per log entry i < L forms the
//             projection coefficients  c^k_i = k^T D(ell' - Lambda_i) K_i,
//             c^q_i = q^T D(...) K_i  (DeltaLog notes Sec. 2.4, warp-shuffle sums), and
//             the L2 norms of q and k (and q_scale) give two per-head scale factors.
//   phase 1   one pass over the tile as chunks land, on the raw vectors:
//             r_k = S^T (e^{ell'} * k),  r_q = S^T (e^{ell'} * q)  (warp-local sums,
//             then across warps), scaled by the norm factors afterwards.
//   phase 2   per value column j:  vhat = r_k + sum_i c^k_i U_i,  b = beta (v - vhat),
//             o = r_q + sum_i c^q_i U_i + (q.k) b.   Append commits the new entry.
//   phase 3   dense / merge only: S' = D(ell') S + sum_i D(ell' - Lambda_i) K_i U_i^T + k b^T,
//             written back with 16-byte coalesced stores.
#include <atomic>

#include "gdn_device.cuh"

namespace gdn {
namespace {

// Two fp32 lanes in one 64-bit register for the packed FMA (fma.rn.f32x2): one
// instruction, two FMAs, each rounded as fmaf rounds.
using f2 = unsigned long long;
__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
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

// Shared-memory layout of one decode CTA (bytes). Identical on host and device.
struct Layout {
  uint32_t tile, bars, scal, vec, uni, us, kd, coef, total;
  int cp;  // row stride (entries) of the merge coefficient table, multiple of 8
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1u) / a * a; }

// Merge forms.  FORM_GENERAL serves every mode and shape.  The three-per-SM merge forms
// (C <= 8, 128-wide heads) fit three CTAs to an SM like dense and append: their U entries go
// to registers (each thread the four columns it folds, the q-owning threads their readout
// column) instead of shared memory.  Under a per-head decay (FORM_R3) ell' takes one entry;
// under a per-key decay (FORM_R3_PER_KEY) e^{ell'} q and e^{ell'} k are not stored but formed
// where phase 1 reads them (the same products, so the same bits).
constexpr int FORM_GENERAL = 0, FORM_R3 = 1, FORM_R3_PER_KEY = 2;

__host__ __device__ inline Layout decode_layout(int mode, int D, int C, int dlam, int klog_bytes, int ulog_bytes,
                                                int form) {
  const bool r3 = form != FORM_GENERAL;
  Layout L{};
  const bool has_log = mode != MODE_DENSE;
  const bool can_merge = mode == MODE_MERGE || mode == MODE_STEP;
  const bool writes_state = mode != MODE_APPEND;
  // the merge folds the log in groups of 8 entries (zero-padded); the current token's
  // term is applied on its own after them
  L.cp = can_merge ? static_cast<int>(align_up(static_cast<uint32_t>(C > 0 ? C : 1), 8u)) : 0;
  uint32_t off = 0;
  L.tile = off;
  off += static_cast<uint32_t>(D * D * 4);
  L.bars = off;
  off += 64;
  L.scal = off;
  off += 128;
  // q (later b), k, q*dec, k*dec, ell', [dec]; FORM_R3: q, k, q*dec, k*dec, dec, ell' (d_lambda
  // entries); FORM_R3_PER_KEY: q, k, dec, ell'.  (The per-key form launches only with
  // d_lambda > 1; the test stays a run-time one, like `ureg` in the kernel: that instance
  // measured about 10% faster so.)
  L.vec = off;
  if (form == FORM_R3_PER_KEY && dlam > 1)
    off += static_cast<uint32_t>(D * 4 * 4);
  else
    off += static_cast<uint32_t>(D * 4 * (writes_state ? 5 : 4)) +
           (r3 ? align_up(static_cast<uint32_t>(dlam * 4), 16u) : static_cast<uint32_t>(D * 4));
  // K_log entries while the coefficients are formed, then the cross-warp partial sums.
  const uint32_t kbytes = has_log ? static_cast<uint32_t>(C * D * klog_bytes) : 0u;
  const uint32_t redbytes = static_cast<uint32_t>(8 * D * 4);
  L.uni = off;
  off += align_up(kbytes > redbytes ? kbytes : redbytes, 16u);
  L.us = off;
  const bool ureg = r3 && C <= 8;
  off += (has_log && !ureg) ? align_up(static_cast<uint32_t>((can_merge ? L.cp : C) * D * ulog_bytes), 16u) : 0u;
  L.kd = off;
  off += can_merge ? static_cast<uint32_t>(D * L.cp * 4) : 0u;
  L.coef = off;  // c^k | c^q | per-head decay snapshots Lambda_i
  off += has_log ? align_up(static_cast<uint32_t>(3 * C * 4), 16u) : 0u;
  L.total = off;
  return L;
}

// The auto step carries both paths; its register cap keeps two CTAs per SM (its shared
// memory allows two).  The three-per-SM merge forms (layout above) cap registers for three:
// with a third CTA resident, the fold's arithmetic hides behind the other CTAs' copies.  The
// other instances take no minimum (0: none).  EXT instances carry the KDA gate
// parametrisation and output epilogue; the others compile them out.
template <int D, int MODE, bool EXT, int FORM>
__global__ void __launch_bounds__(NT_DECODE, FORM != FORM_GENERAL ? 3 : (MODE == MODE_STEP ? 2 : 0))
    gdn_decode_kernel(const DecodeParams p) {
  static_assert(FORM == FORM_GENERAL || MODE == MODE_MERGE || MODE == MODE_STEP,
                "the three-per-SM forms are merge forms (also in the auto step)");
  constexpr bool R3 = FORM != FORM_GENERAL;
  extern __shared__ __align__(128) unsigned char smem[];

  constexpr int NCHUNK = (D >= 128) ? 4 : 1;       // TMA row chunks of the tile
  constexpr int CHUNK_ROWS = D / NCHUNK;
  constexpr uint32_t CHUNK_BYTES = CHUNK_ROWS * D * 4;
  constexpr int VPR = D / 4;                        // float4 per tile row
  constexpr int RPW = 32 / VPR;                     // rows a warp covers per pass
  constexpr int RPI = NW * RPW;                     // rows the CTA covers per pass
  constexpr int NIT = (D + RPI - 1) / RPI;
  constexpr int ITC = NIT / NCHUNK;                 // passes per chunk
  static_assert(NCHUNK == 1 || (NIT % NCHUNK == 0 && CHUNK_ROWS % RPI == 0), "chunking");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool ctrl = warp == NW;  // the copy-issuing warp; warps 0..NW-1 compute
  const int b = blockIdx.x / p.H;
  const int h = blockIdx.x - b * p.H;

  // Launched with programmatic stream serialisation: the first resident wave of CTAs may
  // start while the previous launch in the stream is finishing.  Until griddep_wait() a
  // CTA reads nothing that launch may write and only warms L2: the slot is read as a hint
  // (bounds-checked, used for the prefetch address alone) and the state tile prefetched,
  // so the tail of the previous grid overlaps this grid's first HBM reads.  Later waves
  // start after the previous grid has ended; for them the prefetch would only duplicate
  // their tile copy.
  if (ctrl && lane == 0 && static_cast<int>(blockIdx.x) < p.prefetch_ahead) {
    const int hint = *static_cast<const volatile int*>(p.slot + b);
    if (hint >= 0 && hint < p.num_slots)
      bulk_prefetch_l2(p.state + (static_cast<size_t>(hint) * p.H + h) * static_cast<size_t>(D * D),
                       static_cast<uint32_t>(D * D * 4));
  }
  griddep_launch_dependents();
  griddep_wait();

  const int slot = __ldg(p.slot + b);
  if (slot < 0) return;  // padding request
  if (slot >= p.num_slots) {
    if (tid == 0) atomic_status(p.status, GDN_STATUS_BAD_SLOT);
    return;
  }

  const int C = p.C, dlam = p.dlam;
  const uint32_t fl = p.flags;
  const int klb = (fl & GDN_KLOG_FP32) ? 4 : 2;
  const int ulb = (fl & GDN_ULOG_BF16) ? 2 : 4;
  const Layout L = decode_layout(MODE, D, C, dlam, klb, ulb, FORM);
  // U entries in registers.  The host launches the R3 forms only with C <= 8; the test stays a run-time
  // one on purpose: with the shared-memory path compiled in as well, the instance fits its
  // 72 registers without spilling and measured about 8% faster than with it compiled out.
  const bool ureg = R3 && C <= 8;
  // (likewise the per-key form's test of d_lambda: it launches only with d_lambda > 1)
  const bool pk3 = FORM == FORM_R3_PER_KEY && dlam > 1;
  float* tile = reinterpret_cast<float*>(smem + L.tile);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  int* scal_i = reinterpret_cast<int*>(smem + L.scal);             // [0] L on entry, [1] status bits
  float* scal_f = reinterpret_cast<float*>(smem + L.scal + 16);    // [0..7] norm partials, [8] q.k,
                                                                   // [12..15] output-norm partials
  float* q_s = reinterpret_cast<float*>(smem + L.vec);
  float* b_s = q_s;  // b takes q's place once the prologue is done
  float* k_s = q_s + D;
  float* qdec_s = q_s + 2 * D;
  float* kdec_s = q_s + 3 * D;
  float* ellp_s = q_s + (pk3 ? 3 : (R3 ? 5 : 4)) * D;  // (R3: d_lambda entries, last)
  float* dec_s = q_s + (pk3 ? 2 : (R3 ? 4 : 5)) * D;   // only when the state is written
  unsigned char* uni = smem + L.uni;
  float* red = reinterpret_cast<float*>(uni);
  float* u_s = reinterpret_cast<float*>(smem + L.us);  // U entries (fp32, or bf16 bits)
  uint16_t* u16_s = reinterpret_cast<uint16_t*>(smem + L.us);
  float* kd_s = reinterpret_cast<float*>(smem + L.kd);
  float* ck_s = reinterpret_cast<float*>(smem + L.coef);
  float* cq_s = ck_s + C;
  float* lam_s = ck_s + 2 * C;
  const int cp = L.cp;

  const size_t sh = static_cast<size_t>(slot) * p.H + h;
  const float* tile_g = p.state + sh * static_cast<size_t>(D * D);

  // ---- prologue -------------------------------------------------------------------
  // One lane of the copy-issuing warp starts the tile copy (4 row chunks), the L2
  // prefetch of a later CTA's inputs and, once L has been read, the copy of the first
  // L log entries; the compute warps meanwhile load q/k/v (or run the width-4 conv +
  // SiLU) and form the decays.
  const bool is_q = tid < D;                     // owns q[tid], v[tid], row tid, column tid
  const bool is_k = tid >= 128 && tid < 128 + D;  // owns k[tid - 128]
  const int ii = is_q ? tid : tid - 128;
  float x = 0.0f, vj = 0.0f;
  if (ctrl) {
    const int n_raw = (MODE != MODE_DENSE && lane == 0) ? p.len[sh] : 0;
    if (lane == 0) {
      for (int c = 0; c < NCHUNK; ++c) mbar_init(&bars[c], 1u);
      mbar_init(&bars[NCHUNK], 32u);  // log entries: one cp.async arrival per lane
      fence_mbar_init();
      const uint64_t pol = l2_policy_evict_first();
      const uint32_t starve = (fl & GDN_TEST_STARVE_WAIT) ? 16u : 0u;
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) {
        mbar_arrive_expect_tx(&bars[c], CHUNK_BYTES + (c == 0 ? starve : 0u));
        bulk_load_hint(tile + c * CHUNK_ROWS * D, tile_g + c * CHUNK_ROWS * D, CHUNK_BYTES, &bars[c],
                       pol);
      }
    }
    __syncwarp();  // the log barrier is initialised
    if (MODE != MODE_DENSE) {
      // A merge replays the whole log (L = C), so it copies all C entries at once; the
      // other modes copy the first L as soon as L has been read (entries past L are
      // stale and never read).
      int nc = C;
      if (MODE != MODE_MERGE) {
        nc = __shfl_sync(0xffffffffu, n_raw, 0);
        nc = nc < 0 ? 0 : (nc > C ? C : nc);
      }
      const uint4* ksrc = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.k_log) +
                                                         sh * C * D * klb);
      const uint4* usrc = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.u_log) +
                                                         sh * C * D * ulb);
      const int kvec = nc * D * klb / 16, uvec = nc * D * ulb / 16;
      for (int i = lane; i < kvec; i += 32) cp_async16(reinterpret_cast<uint4*>(uni) + i, ksrc + i);
      if (!ureg)
        for (int i = lane; i < uvec; i += 32) cp_async16(reinterpret_cast<uint4*>(u_s) + i, usrc + i);
      if (dlam == 1)
        for (int e = lane; e < nc; e += 32) cp_async4(lam_s + e, p.lam_log + sh * C + e);
      else if (lane < nc)  // per-key snapshots stay in global memory: warm L2 for the replay
        bulk_prefetch_l2(p.lam_log + (sh * C + lane) * dlam, static_cast<uint32_t>(dlam * 4));
      cp_async_arrive(&bars[NCHUNK]);
    }
    if (lane == 0) {
      // the CTA that runs about one resident wave later finds its token inputs in L2
      // (they depend only on (request, head); the state tile depends on the slot)
      const int gp = static_cast<int>(blockIdx.x) + p.prefetch_ahead;
      if (p.prefetch_ahead > 0 && gp < p.B * p.H) {
        const int bp = gp / p.H, hp = gp - bp * p.H;
        const uint32_t ie = (fl & GDN_QKV_BF16) ? 2u : 4u;
        const uint32_t rowb = static_cast<uint32_t>(D) * ie;
        if (fl & GDN_FUSE_CONV) {
          const unsigned char* row = static_cast<const unsigned char*>(p.mixed) +
                                     static_cast<size_t>(bp) * p.channels * ie;
          const size_t HD = static_cast<size_t>(p.H) * D;
          bulk_prefetch_l2(row + static_cast<size_t>(hp) * D * ie, rowb);
          bulk_prefetch_l2(row + (HD + static_cast<size_t>(hp) * D) * ie, rowb);
          bulk_prefetch_l2(row + (2 * HD + static_cast<size_t>(hp) * D) * ie, rowb);
        } else {
          const size_t off = static_cast<size_t>(gp) * D * ie;
          bulk_prefetch_l2(static_cast<const unsigned char*>(p.q) + off, rowb);
          bulk_prefetch_l2(static_cast<const unsigned char*>(p.k) + off, rowb);
          bulk_prefetch_l2(static_cast<const unsigned char*>(p.v) + off, rowb);
        }
      }
      if (MODE != MODE_DENSE) {
        int n0 = n_raw;
        uint32_t bad0 = 0u;
        if (n0 < 0 || n0 > C)
          bad0 = GDN_STATUS_BAD_LEN;
        else if (MODE == MODE_APPEND && n0 == C)
          bad0 = GDN_STATUS_LOG_FULL;
        if (bad0) n0 = 0;
        scal_i[0] = n0;
        scal_i[1] = static_cast<int>(bad0);
      }
    }
  }
  // both owners of key row ii form its decay exp(ell'), ell' = ell + lambda (closure
  // of the decays; a per-head decay reads entry 0).  The gate loads are issued before
  // the token loads so that the two latencies overlap.
  float lam_t = 0.0f, ell_t = 0.0f, beta = 0.0f, ga = 0.0f, gdt = 0.0f, og = 0.0f;
  if (is_q || is_k) {
    const int di = dlam == 1 ? 0 : ii;
    lam_t = __ldg(p.lam + (static_cast<size_t>(b) * p.H + h) * dlam + di);
    if (MODE != MODE_DENSE) ell_t = p.ell[sh * dlam + di];
    if (EXT && (fl & GDN_GATE_KDA)) {
      ga = __ldg(p.a_log + h);
      gdt = __ldg(p.dt_bias + static_cast<size_t>(h) * dlam + di);
    }
  }
  if ((EXT && (fl & GDN_OUT_NORM_GATE)) && is_q) og = __ldg(p.out_gate + (static_cast<size_t>(b) * p.H + h) * D + ii);
  // U entries in registers: the q-owning threads fetch their readout column of every entry
  // now (only the entries below L enter the readout)
  float ucol[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) ucol[e] = 0.0f;
  if (ureg && is_q) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (e < C) {
        const size_t at = (sh * C + e) * D + tid;
        ucol[e] = (ulb == 2) ? bf16_bits_to_float(static_cast<const uint16_t*>(p.u_log)[at])
                             : static_cast<const float*>(p.u_log)[at];
      }
    }
  }
  if (!ctrl) {
    beta = p.beta ? __ldg(p.beta + static_cast<size_t>(b) * p.H + h) : 1.0f;
    load_token(p, b, h, slot, tid, &x, &vj);
    if (fl & GDN_GATE_RAW) {
      lam_t = log_sigmoidf_(lam_t);
      if (p.beta) beta = sigmoidf_(beta);
    } else if (EXT && (fl & GDN_GATE_KDA)) {
      // KDA gate parametrisation: lambda in (lower_bound, 0), beta = sigmoid(logit)
      lam_t = p.lower_bound * sigmoidf_(expf(ga) * (lam_t + gdt));
      if (p.beta) beta = sigmoidf_(beta);
    }
    const float ss = warp_sum(x * x);
    if (lane == 0) scal_f[warp] = ss;
  }
  const float ellp = ell_t + lam_t;
  if (is_q) {
    const float dcy = expf(ellp);
    q_s[ii] = x;
    if (!pk3) qdec_s[ii] = x * dcy;
    if (MODE != MODE_APPEND) dec_s[ii] = dcy;
    if (ii < dlam) ellp_s[ii] = ellp;
  } else if (is_k) {
    k_s[ii] = x;
    if (!pk3) kdec_s[ii] = x * expf(ellp);
  }
  __syncthreads();  // (A) raw and decayed q, k, decays, norm partials, L and status bits
  if (ctrl) return;  // from here on only the compute warps (named barrier 1)

  const int n = (MODE == MODE_DENSE) ? 0 : scal_i[0];
  const uint32_t bad = (MODE == MODE_DENSE) ? 0u : static_cast<uint32_t>(scal_i[1]);
  if (bad) {  // skip the slot-head: wait for this CTA's own copies, then leave
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) (void)mbar_wait(&bars[c], 0u);
    (void)mbar_wait(&bars[NCHUNK], 0u);
    if (tid == 0) atomic_status(p.status, bad);
    return;
  }
  float kinv = 1.0f, qsc = 1.0f;
  auto norms = [&]() {
    const float qss = scal_f[0] + scal_f[1] + scal_f[2] + scal_f[3];
    const float kss = scal_f[4] + scal_f[5] + scal_f[6] + scal_f[7];
    const bool l2 = (fl & GDN_NO_QK_L2NORM) == 0u;
    kinv = l2 ? 1.0f / sqrtf(kss + p.l2_eps) : 1.0f;
    qsc = (l2 ? 1.0f / sqrtf(qss + p.l2_eps) : 1.0f) * p.q_scale;
  };

  const bool is_merge = (MODE == MODE_MERGE) || (MODE == MODE_STEP && n == C);
  const bool is_append = (MODE == MODE_APPEND) || (MODE == MODE_STEP && n < C);
  bool timeout = false;

  // q.k of the raw vectors (the last warp has the fewest log entries to replay)
  auto qk_dot = [&]() {
    if (warp != NW - 1) return;
    float t = 0.0f;
#pragma unroll
    for (int d = lane; d < D; d += 32) t = fmaf(q_s[d], k_s[d], t);
    t = warp_sum(t);
    if (lane == 0) scal_f[8] = t;
  };

  // log replay coefficients: one warp per entry, w_i = D(ell' - Lambda_i) K_i,
  // c^k_i = k.w_i, c^q_i = q.w_i (warp-shuffle sums); needs only q, k and the log
  auto replay_coefficients = [&]() {
    if (MODE == MODE_DENSE) return;
    // per-key decay: the warp's first entry's snapshot row (warmed in L2) is loaded before
    // the wait for the log copy, so the two latencies overlap
    constexpr int NID = (D + 31) / 32;
    float lpre[NID];
#pragma unroll
    for (int i = 0; i < NID; ++i) lpre[i] = 0.0f;
    if (dlam > 1 && warp < n) {
#pragma unroll
      for (int i = 0; i < NID; ++i) {
        const int d = lane + 32 * i;
        if (d < D) lpre[i] = __ldg(p.lam_log + (sh * C + warp) * dlam + d);
      }
    }
    // wait for the log copy even when L = 0 (a merge copies all C entries), and pad
    // the merge tables only after it
    if (!mbar_wait(&bars[NCHUNK], 0u)) timeout = true;
    if (is_merge) {
      // pad the weight table and the U entries past L with zeros (the group of 8 that
      // holds entry L-1 reads them; the current token's term is applied on its own)
      for (int idx = tid; idx < D * cp; idx += NT) {
        const int d = idx / cp, e = idx - d * cp;
        if (e >= n) kd_s[d * cp + e] = 0.0f;
      }
      if (!ureg) {
        const int pad_words = (cp - n) * D * ulb / 4;
        uint32_t* upad = reinterpret_cast<uint32_t*>(smem + L.us + static_cast<size_t>(n) * D * ulb);
        for (int idx = tid; idx < pad_words; idx += NT) upad[idx] = 0u;
      }
    }
    for (int e = warp; e < n; e += NW) {
      const float* lam_e = p.lam_log + (sh * C + e) * dlam;
      // a per-head decay is one factor of the entry, applied to the two sums
      const float fscal = (dlam == 1) ? expf(ellp_s[0] - lam_s[e]) : 1.0f;
      float ck = 0.0f, cq = 0.0f;
#pragma unroll
      for (int i = 0; i < (D + 31) / 32; ++i) {
        const int d = lane + 32 * i;
        if (d < D) {
          const float kv = (klb == 2)
                               ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(uni)[e * D + d])
                               : reinterpret_cast<const float*>(uni)[e * D + d];
          const float lam_d = (e == warp) ? lpre[i] : __ldg(lam_e + d);
          const float wd = (dlam == 1) ? kv : expf(ellp_s[d] - lam_d) * kv;
          ck = fmaf(k_s[d], wd, ck);
          cq = fmaf(q_s[d], wd, cq);
          if (is_merge) kd_s[d * cp + e] = (dlam == 1) ? fscal * kv : wd;
        }
      }
      ck = warp_sum(ck);
      cq = warp_sum(cq);
      if (lane == 0) {
        ck_s[e] = ck * fscal * kinv;
        cq_s[e] = cq * fscal * qsc;
      }
    }
  };

  // the log was copied from the start; the norm scales, q.k and the replay
  // coefficients are formed while the first tile chunks are still in flight
  norms();
  replay_coefficients();
  qk_dot();

  // ---- phase 1: r_k = S^T (e^{ell'} k), r_q = S^T (e^{ell'} q), one pass --------
  const int c4 = lane % VPR, rsub = lane / VPR;
  const float4* tile4 = reinterpret_cast<const float4*>(tile);
  float ak[4] = {0.f, 0.f, 0.f, 0.f}, aq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < NCHUNK; ++c) {
    if (!mbar_wait(&bars[c], 0u)) timeout = true;
#pragma unroll
    for (int it = c * ITC; it < (c + 1) * ITC; ++it) {
      const int r = it * RPI + warp * RPW + rsub;
      if (r < D) {
        const float4 s = tile4[r * VPR + c4];
        const float kd = pk3 ? k_s[r] * dec_s[r] : kdec_s[r], qd = pk3 ? q_s[r] * dec_s[r] : qdec_s[r];
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
    // the replay coefficients fill the wait for the last chunk
  }
  if (MODE != MODE_DENSE) consumer_sync();  // the K entries share space with the partial sums
#pragma unroll
  for (int off = VPR; off < 32; off <<= 1) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      ak[m] += __shfl_xor_sync(0xffffffffu, ak[m], off);
      aq[m] += __shfl_xor_sync(0xffffffffu, aq[m], off);
    }
  }
  // across warps, fixed order: red[w] = part[w + 4] + part[w], then sum over w
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
  // the step goes ahead: only now does the conv cache row shift (a call that timed out
  // above has written nothing, the cache included, so retrying it is safe)
  if (fl & GDN_FUSE_CONV) conv_commit(p, b, h, slot, tid);

  // ---- phase 2: residual, write strength, readout, log commit ----------------------
  float oj = 0.0f;
  if (is_q) {
    const int j = tid;
    float rk = red[j];
    rk += red[2 * D + j];
    rk += red[4 * D + j];
    rk += red[6 * D + j];
    float rq = red[D + j];
    rq += red[3 * D + j];
    rq += red[5 * D + j];
    rq += red[7 * D + j];
    // the sums ran on the raw vectors; an explicit rounded product keeps every mode
    // (with or without log terms after it) on the same arithmetic
    rk = __fmul_rn(rk, kinv);
    rq = __fmul_rn(rq, qsc);
    if (ureg) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e < n) {
          rk = fmaf(ck_s[e], ucol[e], rk);
          rq = fmaf(cq_s[e], ucol[e], rq);
        }
      }
    } else {
      for (int e = 0; e < n; ++e) {
        const float u = (ulb == 2) ? bf16_bits_to_float(u16_s[e * D + j]) : u_s[e * D + j];
        rk = fmaf(ck_s[e], u, rk);
        rq = fmaf(cq_s[e], u, rq);
      }
    }
    const float bj = (fl & GDN_PLAIN_UPDATE) ? beta * vj : beta * (vj - rk);
    oj = fmaf(scal_f[8] * qsc * kinv, bj, rq);
    if (!(EXT && (fl & GDN_OUT_NORM_GATE))) p.o[(static_cast<size_t>(b) * p.H + h) * D + j] = oj;
    b_s[j] = bj;
    if (is_append) {
      const float uval = (fl & GDN_KLOG_PRENORM) ? bj * kinv : bj;
      const size_t at = (sh * C + n) * D + j;
      if (ulb == 2)
        reinterpret_cast<__nv_bfloat16*>(p.u_log)[at] = __float2bfloat16_rn(uval);
      else
        static_cast<float*>(p.u_log)[at] = uval;
    }
  }
  if (EXT && (fl & GDN_OUT_NORM_GATE)) {
    // KDA output epilogue: o <- o / sqrt(mean(o^2) + eps) * w * sigmoid(g) over the head's
    // dv channels (the q-owning warps 0..3 hold them; the other lanes add zero)
    const float ss = warp_sum(oj * oj);
    if (lane == 0 && warp < 4) scal_f[12 + warp] = ss;
    consumer_sync();
    if (is_q) {
      const float ms = (scal_f[12] + scal_f[13] + scal_f[14] + scal_f[15]) / static_cast<float>(D);
      const float w = p.out_norm_w ? __ldg(p.out_norm_w + tid) : 1.0f;
      p.o[(static_cast<size_t>(b) * p.H + h) * D + tid] = oj * (1.0f / sqrtf(ms + p.out_eps)) * w * sigmoidf_(og);
    }
  }
  if (is_append) {
    if (is_k) {
      const float kval = (fl & GDN_KLOG_PRENORM) ? x : x * kinv;
      const size_t at = (sh * C + n) * D + ii;
      if (klb == 2)
        reinterpret_cast<__nv_bfloat16*>(p.k_log)[at] = __float2bfloat16_rn(kval);
      else
        reinterpret_cast<float*>(p.k_log)[at] = kval;
    }
    if (tid < dlam) {
      p.lam_log[(sh * C + n) * dlam + tid] = ellp_s[tid];
      p.ell[sh * dlam + tid] = ellp_s[tid];
    }
    if (tid == 0) p.len[sh] = n + 1;
  } else if (is_merge) {
    if (tid < dlam) p.ell[sh * dlam + tid] = 0.0f;
    if (tid == 0) p.len[sh] = 0;
  }

  // ---- phase 3: write the state (dense) or fold the log into the base (merge) ------
  // S' = D(ell') S + sum_{i<L} (e^{ell' - Lambda_i} K_i) U_i^T + k b^T: the log terms in
  // groups of 8 (zero-padded), then the current token's term, in that order; with L = 0
  // this is the dense arithmetic exactly.
  if (MODE == MODE_DENSE || is_merge) {
    consumer_sync();  // (F) b and the padded tables are in shared memory
    float* out = p.state + sh * static_cast<size_t>(D * D);
    float4* tilew = reinterpret_cast<float4*>(tile);
    const float4 bb = reinterpret_cast<const float4*>(b_s)[c4];
    const int ng = (MODE == MODE_DENSE) ? 0 : (n + 7) / 8;
    for (int g = 0; g < ng; ++g) {
      float4 u[8];
      if (ureg) {
        // this thread's four columns of each entry, from global memory (the lines the
        // readout-column fetch brought in); zero past L
        const unsigned char* ub = static_cast<const unsigned char*>(p.u_log) + sh * C * D * ulb;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          u[e] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (e < n) {
            if (ulb == 2) {
              const uint2 raw = reinterpret_cast<const uint2*>(ub + static_cast<size_t>(e) * D * 2)[c4];
              u[e] = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                                 __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
            } else {
              u[e] = reinterpret_cast<const float4*>(ub + static_cast<size_t>(e) * D * 4)[c4];
            }
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (ulb == 2) {
            const uint2 raw = reinterpret_cast<const uint2*>(u16_s + (g * 8 + e) * D)[c4];
            u[e] = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                               __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
          } else {
            u[e] = reinterpret_cast<const float4*>(u_s + (g * 8 + e) * D)[c4];
          }
        }
      }
      // (R3 folds with packed FMAs on column pairs: the same roundings, fewer instructions)
      f2 u01[8], u23[8];
      if (R3) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          u01[e] = f2_pack(u[e].x, u[e].y);
          u23[e] = f2_pack(u[e].z, u[e].w);
        }
      }
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        const int r = it * RPI + warp * RPW + rsub;
        if (r < D) {
          float4 acc = tile4[r * VPR + c4];
          if (g == 0) {
            const float dc = dec_s[r];
            acc.x *= dc;
            acc.y *= dc;
            acc.z *= dc;
            acc.w *= dc;
          }
          const float4 w0 = *reinterpret_cast<const float4*>(kd_s + r * cp + g * 8);
          const float4 w1 = *reinterpret_cast<const float4*>(kd_s + r * cp + g * 8 + 4);
          const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          if (R3) {
            f2 a01 = f2_pack(acc.x, acc.y), a23 = f2_pack(acc.z, acc.w);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const f2 ws = f2_pack(wv[e], wv[e]);
              a01 = f2_fma(ws, u01[e], a01);
              a23 = f2_fma(ws, u23[e], a23);
            }
            f2_unpack(a01, acc.x, acc.y);
            f2_unpack(a23, acc.z, acc.w);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              acc.x = fmaf(wv[e], u[e].x, acc.x);
              acc.y = fmaf(wv[e], u[e].y, acc.y);
              acc.z = fmaf(wv[e], u[e].z, acc.z);
              acc.w = fmaf(wv[e], u[e].w, acc.w);
            }
          }
          if (g == ng - 1) {  // the current token's term, then the write-back
            const float kk = k_s[r] * kinv;
            acc.x = fmaf(kk, bb.x, acc.x);
            acc.y = fmaf(kk, bb.y, acc.y);
            acc.z = fmaf(kk, bb.z, acc.z);
            acc.w = fmaf(kk, bb.w, acc.w);
            *reinterpret_cast<float4*>(out + r * D + c4 * 4) = acc;
          } else {
            tilew[r * VPR + c4] = acc;
          }
        }
      }
    }
    if (ng == 0) {  // dense, or a merge of an empty log
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
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------
// launchers


constexpr int kMaxDevices = 64;

int sm_count(int dev) {
  static std::atomic<int> cache[kMaxDevices];
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}


template <int D, int MODE, bool EXT, int FORM>
cudaError_t launch_one(const DecodeParams& p, cudaStream_t stream) {
  static std::atomic<uint32_t> configured[kMaxDevices];
  const int klb = (p.flags & GDN_KLOG_FP32) ? 4 : 2;
  const int ulb = (p.flags & GDN_ULOG_BF16) ? 2 : 4;
  const Layout L = decode_layout(MODE, D, p.C, p.dlam, klb, ulb, FORM);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (configured[dev].load(std::memory_order_relaxed) < L.total) {
    err = cudaFuncSetAttribute(gdn_decode_kernel<D, MODE, EXT, FORM>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(L.total));
    if (err != cudaSuccess) return err;
    // several 64 KiB-tile CTAs per SM only fit with the whole L1/shared array as shared memory
    err = cudaFuncSetAttribute(gdn_decode_kernel<D, MODE, EXT, FORM>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (err != cudaSuccess) return err;
    configured[dev].store(L.total, std::memory_order_relaxed);
  }
  // prefetch distance for the token inputs: the number of CTAs resident at once
  // (cached per device as (shared bytes << 32 | CTAs per SM))
  static std::atomic<uint64_t> resident[kMaxDevices];
  uint64_t rc = resident[dev].load(std::memory_order_relaxed);
  if ((rc >> 32) != L.total) {
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gdn_decode_kernel<D, MODE, EXT, FORM>, NT_DECODE,
                                                        L.total);
    if (err != cudaSuccess) return err;
    rc = (static_cast<uint64_t>(L.total) << 32) | static_cast<uint32_t>(per_sm > 0 ? per_sm : 1);
    resident[dev].store(rc, std::memory_order_relaxed);
  }
  DecodeParams q = p;
  q.prefetch_ahead = static_cast<int>(rc & 0xffffffffu) * sm_count(dev);
  // programmatic stream serialisation: the kernel orders its own reads (griddep_wait)
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
  err = cudaLaunchKernelEx(&cfg, gdn_decode_kernel<D, MODE, EXT, FORM>, q);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// The form a merge of a 128-wide head takes: a three-per-SM form when C <= 8, the U log is
// fp32 and its layout fits three CTAs in the SM's shared memory (each CTA also takes the
// per-block reservation); otherwise the general form, two CTAs per SM without the register
// cap.  (A bf16 U log unpacks every entry in the fold: the one such workload, RWKV6, measured
// its merge 5% slower in the three-per-SM form.)
int merge_form(const DecodeParams& p) {
  if (p.D != 128 || p.C > 8 || (p.flags & GDN_ULOG_BF16)) return FORM_GENERAL;
  const int form = p.dlam == 1 ? FORM_R3 : FORM_R3_PER_KEY;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FORM_GENERAL;
  static std::atomic<int> budget[kMaxDevices];
  int b = budget[dev].load(std::memory_order_relaxed);
  if (b == 0) {
    int per_sm = 0, reserved = 0;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
      return FORM_GENERAL;
    b = per_sm / 3 - reserved;
    budget[dev].store(b > 0 ? b : -1, std::memory_order_relaxed);
  }
  const int klb = (p.flags & GDN_KLOG_FP32) ? 4 : 2;
  const int ulb = (p.flags & GDN_ULOG_BF16) ? 2 : 4;
  const bool fits = b > 0 && decode_layout(MODE_MERGE, 128, p.C, p.dlam, klb, ulb, form).total <= static_cast<uint32_t>(b);
  return fits ? form : FORM_GENERAL;
}

template <int D, bool EXT>
cudaError_t launch_de(int mode, const DecodeParams& p, cudaStream_t stream) {
  switch (mode) {
    case MODE_DENSE: return launch_one<D, MODE_DENSE, EXT, FORM_GENERAL>(p, stream);
    case MODE_APPEND: return launch_one<D, MODE_APPEND, EXT, FORM_GENERAL>(p, stream);
    case MODE_MERGE:
      if constexpr (D == 128) {
        switch (merge_form(p)) {
          case FORM_R3: return launch_one<D, MODE_MERGE, EXT, FORM_R3>(p, stream);
          case FORM_R3_PER_KEY: return launch_one<D, MODE_MERGE, EXT, FORM_R3_PER_KEY>(p, stream);
          default: break;
        }
      }
      return launch_one<D, MODE_MERGE, EXT, FORM_GENERAL>(p, stream);
    case MODE_STEP:
      if constexpr (D == 128) {
        switch (merge_form(p)) {
          case FORM_R3: return launch_one<D, MODE_STEP, EXT, FORM_R3>(p, stream);
          case FORM_R3_PER_KEY: return launch_one<D, MODE_STEP, EXT, FORM_R3_PER_KEY>(p, stream);
          default: break;
        }
      }
      return launch_one<D, MODE_STEP, EXT, FORM_GENERAL>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_d(int mode, const DecodeParams& p, cudaStream_t stream) {
  if (p.flags & (GDN_GATE_KDA | GDN_OUT_NORM_GATE)) return launch_de<D, true>(mode, p, stream);
  return launch_de<D, false>(mode, p, stream);
}

}  // namespace

size_t decode_smem_bytes(int mode, int dk, int dv, int ns, int C, int dlam, int klog_bytes, int ulog_bytes) {
  if (!decode_shape_built(dk, dv, ns)) return 0;
  if (ns == 1 && dk == dv) return decode_layout(mode, dk, C, dlam, klog_bytes, ulog_bytes, FORM_GENERAL).total;
  return decode_smem_bytes_x(mode, dk, dv, ns, C, klog_bytes, ulog_bytes);
}

bool decode_shape_built(int dk, int dv, int ns) {
  if (ns == 1)
    return (dk == dv && (dk == 16 || dk == 32 || dk == 64 || dk == 128)) || (dk == 128 && dv == 64) ||
           (dk == 64 && dv == 128);
  if (ns == 2) return dk == dv && (dk == 64 || dk == 128);
  return false;
}

cudaError_t launch_decode(int mode, const DecodeParams& p, cudaStream_t stream) {
  if ((p.flags & GDN_SPLIT_DV) == 0u && p.D == p.DV) {
    switch (p.D) {
      case 16: return launch_d<16>(mode, p, stream);
      case 32: return launch_d<32>(mode, p, stream);
      case 64: return launch_d<64>(mode, p, stream);
      case 128: return launch_d<128>(mode, p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  return launch_decode_x(mode, p, stream);
}

}  // namespace gdn
