// gdn_decode_kernel.cuh -- the decode-step kernel (dense, DeltaLog append, merge, auto step),
// templated on the key head size DK, the value head size DV and the number NS of CTAs that
// share one (request, head) along dv. gdn_decode_x.cu instantiates it for the shapes the
// square one-CTA kernel of gdn_decode.cu does not cover.
//
// Each CTA owns one value slice of one (request, head): DVS = DV / NS value columns of the
// state tile S[DK][DV] (all of it when NS = 1), the matching columns of the output row and of
// the value log, and is their single writer (DeltaLog notes, Sec. 2.6 / Fig. 5 slice the tile
// along dv). With NS = 2 the two slices of a head run as one cluster: slice 0 is the single
// writer of the head's shared metadata (K_log[L], Lambda_log[L], ell, L) and of the q / k conv
// cache rows, and writes them only after the cluster barrier has seen slice 1 read them.
//
// Per CTA (8 compute warps + 1 copy-issuing warp):
//   launch    programmatic stream serialisation: the CTA lets the next launch schedule at
//             once and waits for the previous grid before its first read (first-wave CTAs
//             prefetch their tile into L2 before that wait).
//   prologue  the copy warp starts the copies of the tile slice (TMA bulk copies of whole
//             rows when NS = 1, 2-D TMA tiles of the slice's columns otherwise) and of the log (append:
//             the first L entries once L is read; merge: all C); the compute warps load the
//             gates and q/k/v (or run the width-4 conv + SiLU) and form the decays
//             exp(ell').  One barrier.
//   replay    while the tile is in flight, one warp per log entry i < L forms the
//             projection coefficients  c^k_i = k^T D(ell' - Lambda_i) K_i,
//             c^q_i = q^T D(...) K_i  (DeltaLog notes Sec. 2.4, warp-shuffle sums), and
//             the L2 norms of q and k (and q_scale) give two per-head scale factors.
//   phase 1   one pass over the tile as chunks land, on the raw vectors:
//             r_k = S^T (e^{ell'} * k),  r_q = S^T (e^{ell'} * q)  (warp-local sums,
//             then across warps), scaled by the norm factors afterwards.
//   phase 2   per value column j of the slice:  vhat = r_k + sum_i c^k_i U_i,
//             b = beta (v - vhat),  o = r_q + sum_i c^q_i U_i + (q.k) b.   Append commits
//             the new entry.
//   phase 3   dense / merge only: S' = D(ell') S + sum_i D(ell' - Lambda_i) K_i U_i^T + k b^T,
//             written back with 16-byte coalesced stores.
#pragma once

#include <atomic>

#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime's driver entry point)

#include "gdn_device.cuh"

namespace gdn {
namespace shaped {

// Shared-memory layout of one decode CTA (bytes). Identical on host and device.
struct Layout {
  uint32_t tile, bars, scal, vec, uni, us, kd, coef, total;
  int cp;  // row stride (entries) of the merge coefficient table, multiple of 8
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1u) / a * a; }

// DK key rows, DVS value columns per CTA. b (DVS values) takes q's place once q is no longer
// needed when it fits there (DVS <= DK), else it has its own vector.
__host__ __device__ inline Layout decode_layout(int mode, int DK, int DVS, int C, int klog_bytes, int ulog_bytes) {
  Layout L{};
  const bool has_log = mode != MODE_DENSE;
  const bool can_merge = mode == MODE_MERGE || mode == MODE_STEP;
  const bool writes_state = mode != MODE_APPEND;
  // the merge folds the log in groups of 8 entries (zero-padded); the current token's
  // term is applied on its own after them
  L.cp = can_merge ? static_cast<int>(align_up(static_cast<uint32_t>(C > 0 ? C : 1), 8u)) : 0;
  uint32_t off = 0;
  L.tile = off;
  off += static_cast<uint32_t>(DK * DVS * 4);
  L.bars = off;
  off += 64;
  L.scal = off;
  off += 128;
  L.vec = off;  // q (later b), k, q*dec, k*dec, ell', [dec] (DK each), [b (DVS)]
  off += static_cast<uint32_t>(DK * 4 * (writes_state ? 6 : 5) + (DVS > DK ? DVS * 4 : 0));
  // K_log entries while the coefficients are formed, then the cross-warp partial sums.
  const uint32_t kbytes = has_log ? static_cast<uint32_t>(C * DK * klog_bytes) : 0u;
  const uint32_t redbytes = static_cast<uint32_t>(8 * DVS * 4);
  L.uni = off;
  off += align_up(kbytes > redbytes ? kbytes : redbytes, 16u);
  L.us = off;
  off += has_log ? align_up(static_cast<uint32_t>((can_merge ? L.cp : C) * DVS * ulog_bytes), 16u) : 0u;
  L.kd = off;
  off += can_merge ? static_cast<uint32_t>(DK * L.cp * 4) : 0u;
  L.coef = off;  // c^k | c^q | per-head decay snapshots Lambda_i
  off += has_log ? align_up(static_cast<uint32_t>(3 * C * 4), 16u) : 0u;
  L.total = off;
  return L;
}

// ---- cluster barrier of the two slices of a head (NS = 2) ----------------------------------
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// waits until every non-exited thread of the cluster has arrived
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// ---- input stage of one (request, head) for DK / DV heads -------------------------------------
// Channel c of the projected token: [q heads (H*DK) | k heads (H*DK) | v heads (H*DV)].
template <int DK, int DV>
__device__ __forceinline__ int qkv_channel(const DecodeParams& p, int which, int h, int i) {
  return which == 0 ? h * DK + i : (which == 1 ? p.H * DK + h * DK + i : 2 * p.H * DK + h * DV + i);
}

// TMA load of one 2-D box of a tensor map (x innermost, in elements) into shared memory,
// completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Tile-copy argument of a launch: nothing when the CTA owns whole rows (NS = 1); for split
// heads the state pool as a 2-D fp32 tensor map of num_slots*H*DK rows and DV columns, boxes
// of CHUNK_ROWS rows by DV/NS columns. (A tensor-map parameter is left out of the other
// launches: it costs every launch its setup.)
template <int NS>
struct TileMap {
  int unused;
};
template <>
struct TileMap<2> {
  CUtensorMap map;
};

// q / k of this thread's key channel (threads [0, DK) and [128, 128 + DK)), v of its value
// column (threads [0, DVS): column col0 + tid). The conv reads the pre-conv cache rows only
// (shifted once the step is known to go ahead). One function, the q / v pair loaded
// together: issued back to back, the v load is not left to wait for its first use.
template <int DK, int DV, int DVS>
__device__ __forceinline__ void load_qkv(const DecodeParams& p, int b, int h, int slot, int tid, int col0, bool conv,
                                         bool bf16, float* x, float* vj) {
  const bool is_q = tid < DK;
  const bool is_k = tid >= 128 && tid < 128 + DK;
  const bool is_col = tid < DVS;
  *x = 0.0f;
  *vj = 0.0f;
  if (!is_q && !is_k && !is_col) return;
  const int i = is_q ? tid : tid - 128;
  if (conv) {
    if (is_q || is_k) *x = conv_silu_channel(p, b, slot, qkv_channel<DK, DV>(p, is_q ? 0 : 1, h, i), bf16);
    if (is_col) *vj = conv_silu_channel(p, b, slot, qkv_channel<DK, DV>(p, 2, h, col0 + tid), bf16);
  } else {
    const size_t hq = static_cast<size_t>(b) * p.H + h;
    if (is_q) {
      *x = load_elem(p.q, hq * DK + i, bf16);
      if (is_col) *vj = load_elem(p.v, hq * DV + col0 + tid, bf16);
    } else if (is_k) {
      *x = load_elem(p.k, hq * DK + i, bf16);
    } else {
      *vj = load_elem(p.v, hq * DV + col0 + tid, bf16);
    }
  }
}

template <int DK, int DV, int NS, int MODE, bool EXT>
__global__ void __launch_bounds__(NT_DECODE, MODE == MODE_STEP ? 2 : 0)
    gdn_decode_kernel(const DecodeParams p, const __grid_constant__ TileMap<NS> tmap) {
  extern __shared__ __align__(128) unsigned char smem[];

  constexpr int DVS = DV / NS;                      // value columns of this CTA
  constexpr int NCHUNK = (DK >= 128) ? 4 : 1;       // row chunks of the tile copy
  constexpr int CHUNK_ROWS = DK / NCHUNK;
  constexpr uint32_t CHUNK_BYTES = CHUNK_ROWS * DVS * 4;
  constexpr int VPR = DVS / 4;                      // float4 per tile row
  constexpr int RPW = 32 / VPR;                     // rows a warp covers per pass
  constexpr int RPI = NW * RPW;                     // rows the CTA covers per pass
  constexpr int NIT = (DK + RPI - 1) / RPI;
  constexpr int ITC = NIT / NCHUNK;                 // passes per chunk
  static_assert(NCHUNK == 1 || (NIT % NCHUNK == 0 && CHUNK_ROWS % RPI == 0), "chunking");
  static_assert(DK <= 128 && DVS <= 128 && VPR >= 1 && VPR <= 32, "head sizes");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool ctrl = warp == NW;  // the copy-issuing warp; warps 0..NW-1 compute
  const int item = NS == 1 ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) / NS;
  const int sl = static_cast<int>(blockIdx.x) - item * NS;  // value slice of this CTA
  const int b = item / p.H;
  const int h = item - b * p.H;
  const bool writer = sl == 0;  // single writer of the head's shared metadata

  // Launched with programmatic stream serialisation: the first resident wave of CTAs may
  // start while the previous launch in the stream is finishing.  Until griddep_wait() a
  // CTA reads nothing that launch may write and only warms L2: the slot is read as a hint
  // (bounds-checked, used for the prefetch address alone) and its share of the state tile
  // prefetched, so the tail of the previous grid overlaps this grid's first HBM reads.
  if (ctrl && lane == 0 && static_cast<int>(blockIdx.x) < p.prefetch_ahead) {
    const int hint = *static_cast<const volatile int*>(p.slot + b);
    if (hint >= 0 && hint < p.num_slots)
      bulk_prefetch_l2(p.state + (static_cast<size_t>(hint) * p.H + h) * static_cast<size_t>(DK * DV) +
                           static_cast<size_t>(sl) * (DK / NS) * DV,
                       static_cast<uint32_t>(DK / NS * DV * 4));
  }
  griddep_launch_dependents();
  griddep_wait();

  const int slot = __ldg(p.slot + b);
  if (slot < 0) return;  // padding request
  if (slot >= p.num_slots) {
    if (tid == 0 && writer) atomic_status(p.status, GDN_STATUS_BAD_SLOT);
    return;
  }

  const int C = p.C, dlam = p.dlam;
  const uint32_t fl = p.flags;
  const int klb = (fl & GDN_KLOG_FP32) ? 4 : 2;
  const int ulb = (fl & GDN_ULOG_BF16) ? 2 : 4;
  const Layout L = decode_layout(MODE, DK, DVS, C, klb, ulb);
  float* tile = reinterpret_cast<float*>(smem + L.tile);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  int* scal_i = reinterpret_cast<int*>(smem + L.scal);             // [0] L on entry, [1] status bits
  float* scal_f = reinterpret_cast<float*>(smem + L.scal + 16);    // [0..7] norm partials, [8] q.k,
                                                                   // [12..15] output-norm partials
  float* q_s = reinterpret_cast<float*>(smem + L.vec);
  float* k_s = q_s + DK;
  float* qdec_s = q_s + 2 * DK;
  float* kdec_s = q_s + 3 * DK;
  float* ellp_s = q_s + 4 * DK;
  float* dec_s = q_s + 5 * DK;                                       // only when the state is written
  float* b_s = DVS <= DK ? q_s : q_s + ((MODE != MODE_APPEND) ? 6 : 5) * DK;  // b of the slice's columns
  unsigned char* uni = smem + L.uni;
  float* red = reinterpret_cast<float*>(uni);
  float* u_s = reinterpret_cast<float*>(smem + L.us);  // U entries of the slice (fp32, or bf16 bits)
  uint16_t* u16_s = reinterpret_cast<uint16_t*>(smem + L.us);
  float* kd_s = reinterpret_cast<float*>(smem + L.kd);
  float* ck_s = reinterpret_cast<float*>(smem + L.coef);
  float* cq_s = ck_s + C;
  float* lam_s = ck_s + 2 * C;
  const int cp = L.cp;

  const size_t sh = static_cast<size_t>(slot) * p.H + h;
  const float* tile_g = p.state + sh * static_cast<size_t>(DK * DV) + static_cast<size_t>(sl) * DVS;
  const int col0 = sl * DVS;  // first value column of the slice

  // ---- prologue -------------------------------------------------------------------------
  const bool is_q = tid < DK;                      // owns q[tid], row tid
  const bool is_k = tid >= 128 && tid < 128 + DK;  // owns k[tid - 128]
  const bool is_col = tid < DVS;                   // owns value column col0 + tid of the slice
  const int ii = is_q ? tid : tid - 128;
  const bool bf16 = (fl & GDN_QKV_BF16) != 0u;
  const bool conv = (fl & GDN_FUSE_CONV) != 0u;
  float x = 0.0f, vj = 0.0f;
  if (ctrl) {
    const int n_raw = (MODE != MODE_DENSE && lane == 0) ? p.len[sh] : 0;
    if (lane == 0) {
      // one TMA copy per row chunk: NS = 1 a bulk copy (the rows are contiguous), NS = 2 a
      // 2-D box of the slice's columns
      const uint32_t starve = (fl & GDN_TEST_STARVE_WAIT) ? 16u : 0u;
      for (int c = 0; c < NCHUNK; ++c) mbar_init(&bars[c], 1u);
      mbar_init(&bars[NCHUNK], 32u);  // log entries: one cp.async arrival per lane
      fence_mbar_init();
      const uint64_t pol = l2_policy_evict_first();
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) {
        mbar_arrive_expect_tx(&bars[c], CHUNK_BYTES + (c == 0 ? starve : 0u));
        if constexpr (NS == 1)
          bulk_load_hint(tile + c * CHUNK_ROWS * DVS, tile_g + c * CHUNK_ROWS * DV, CHUNK_BYTES, &bars[c], pol);
        else
          tma_load_2d(tile + c * CHUNK_ROWS * DVS, &tmap.map, col0, static_cast<int>(sh * DK) + c * CHUNK_ROWS,
                      &bars[c]);
      }
    }
    __syncwarp();  // the barriers are initialised
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
                                                         sh * C * DK * klb);
      const int kvec = nc * DK * klb / 16;
      for (int i = lane; i < kvec; i += 32) cp_async16(reinterpret_cast<uint4*>(uni) + i, ksrc + i);
      // the slice's columns of each U entry (rows of DV values, DVS of them contiguous; one
      // contiguous run of nc rows when the CTA owns all of them)
      const unsigned char* ubase = static_cast<const unsigned char*>(p.u_log) + (sh * C * DV + col0) * ulb;
      if (NS == 1) {
        const int uvec = nc * DV * ulb / 16;
        for (int i = lane; i < uvec; i += 32)
          cp_async16(reinterpret_cast<uint4*>(u16_s) + i, reinterpret_cast<const uint4*>(ubase) + i);
      } else {
        const int upr = DVS * ulb / 16;  // 16-byte pieces per entry row of the slice
        for (int i = lane; i < nc * upr; i += 32) {
          const int e = i / upr, q16 = i - e * upr;
          cp_async16(reinterpret_cast<uint4*>(u16_s) + e * upr + q16,
                     reinterpret_cast<const uint4*>(ubase + static_cast<size_t>(e) * DV * ulb) + q16);
        }
      }
      if (dlam == 1)
        for (int e = lane; e < nc; e += 32) cp_async4(lam_s + e, p.lam_log + sh * C + e);
      else if (lane < nc)  // per-key snapshots stay in global memory: warm L2 for the replay
        bulk_prefetch_l2(p.lam_log + (sh * C + lane) * dlam, static_cast<uint32_t>(dlam * 4));
      cp_async_arrive(&bars[NCHUNK]);
    }
    if (lane == 0) {
      // the CTA that runs about one resident wave later finds its token inputs in L2
      // (they depend only on (request, head); the state tile depends on the slot)
      const int gp = (static_cast<int>(blockIdx.x) + p.prefetch_ahead) / NS;
      if (p.prefetch_ahead > 0 && gp < p.B * p.H) {
        const int bp = gp / p.H, hp = gp - bp * p.H;
        const uint32_t ie = bf16 ? 2u : 4u;
        if (conv) {
          const unsigned char* row = static_cast<const unsigned char*>(p.mixed) +
                                     static_cast<size_t>(bp) * p.channels * ie;
          bulk_prefetch_l2(row + static_cast<size_t>(qkv_channel<DK, DV>(p, 0, hp, 0)) * ie, DK * ie);
          bulk_prefetch_l2(row + static_cast<size_t>(qkv_channel<DK, DV>(p, 1, hp, 0)) * ie, DK * ie);
          bulk_prefetch_l2(row + static_cast<size_t>(qkv_channel<DK, DV>(p, 2, hp, 0)) * ie, DV * ie);
        } else {
          bulk_prefetch_l2(static_cast<const unsigned char*>(p.q) + static_cast<size_t>(gp) * DK * ie, DK * ie);
          bulk_prefetch_l2(static_cast<const unsigned char*>(p.k) + static_cast<size_t>(gp) * DK * ie, DK * ie);
          bulk_prefetch_l2(static_cast<const unsigned char*>(p.v) + static_cast<size_t>(gp) * DV * ie, DV * ie);
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
  if ((EXT && (fl & GDN_OUT_NORM_GATE)) && is_col)
    og = __ldg(p.out_gate + (static_cast<size_t>(b) * p.H + h) * DV + col0 + tid);
  if (!ctrl) {
    beta = p.beta ? __ldg(p.beta + static_cast<size_t>(b) * p.H + h) : 1.0f;
    load_qkv<DK, DV, DVS>(p, b, h, slot, tid, col0, conv, bf16, &x, &vj);
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
    qdec_s[ii] = x * dcy;
    if (MODE != MODE_APPEND) dec_s[ii] = dcy;
    if (ii < dlam) ellp_s[ii] = ellp;
  } else if (is_k) {
    k_s[ii] = x;
    kdec_s[ii] = x * expf(ellp);
  }
  __syncthreads();  // (A) raw and decayed q, k, decays, norm partials, L and status bits
  // every read of the head's shared metadata (L, ell) and of its q / k conv rows lies before
  // this point: the slices of a cluster arrive here, and slice 0 waits for the arrival of
  // slice 1 before it overwrites any of it
  if (NS > 1) cluster_arrive();
  if (ctrl) return;  // from here on only the compute warps (named barrier 1)

  const int n = (MODE == MODE_DENSE) ? 0 : scal_i[0];
  const uint32_t bad = (MODE == MODE_DENSE) ? 0u : static_cast<uint32_t>(scal_i[1]);
  if (bad) {  // skip the slot-head: wait for this CTA's own copies, then leave
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) (void)mbar_wait(&bars[c], 0u);
    (void)mbar_wait(&bars[NCHUNK], 0u);
    if (tid == 0 && writer) atomic_status(p.status, bad);
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
    for (int d = lane; d < DK; d += 32) t = fmaf(q_s[d], k_s[d], t);
    t = warp_sum(t);
    if (lane == 0) scal_f[8] = t;
  };

  // log replay coefficients: one warp per entry, w_i = D(ell' - Lambda_i) K_i,
  // c^k_i = k.w_i, c^q_i = q.w_i (warp-shuffle sums); needs only q, k and the log
  auto replay_coefficients = [&]() {
    if (MODE == MODE_DENSE) return;
    // per-key decay: the warp's first entry's snapshot row (warmed in L2) is loaded before
    // the wait for the log copy, so the two latencies overlap
    constexpr int NID = (DK + 31) / 32;
    float lpre[NID];
#pragma unroll
    for (int i = 0; i < NID; ++i) lpre[i] = 0.0f;
    if (dlam > 1 && warp < n) {
#pragma unroll
      for (int i = 0; i < NID; ++i) {
        const int d = lane + 32 * i;
        if (d < DK) lpre[i] = __ldg(p.lam_log + (sh * C + warp) * dlam + d);
      }
    }
    // wait for the log copy even when L = 0 (a merge copies all C entries), and pad
    // the merge tables only after it
    if (!mbar_wait(&bars[NCHUNK], 0u)) timeout = true;
    if (is_merge) {
      // pad the weight table and the U entries past L with zeros (the group of 8 that
      // holds entry L-1 reads them; the current token's term is applied on its own)
      for (int idx = tid; idx < DK * cp; idx += NT) {
        const int d = idx / cp, e = idx - d * cp;
        if (e >= n) kd_s[d * cp + e] = 0.0f;
      }
      const int pad_words = (cp - n) * DVS * ulb / 4;
      uint32_t* upad = reinterpret_cast<uint32_t*>(smem + L.us + static_cast<size_t>(n) * DVS * ulb);
      for (int idx = tid; idx < pad_words; idx += NT) upad[idx] = 0u;
    }
    for (int e = warp; e < n; e += NW) {
      const float* lam_e = p.lam_log + (sh * C + e) * dlam;
      // a per-head decay is one factor of the entry, applied to the two sums
      const float fscal = (dlam == 1) ? expf(ellp_s[0] - lam_s[e]) : 1.0f;
      float ck = 0.0f, cq = 0.0f;
#pragma unroll
      for (int i = 0; i < (DK + 31) / 32; ++i) {
        const int d = lane + 32 * i;
        if (d < DK) {
          const float kv = (klb == 2)
                               ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(uni)[e * DK + d])
                               : reinterpret_cast<const float*>(uni)[e * DK + d];
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
      if (r < DK) {
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
    float* r0 = red + (warp - 4) * 2 * DVS + c4 * 4;
    *reinterpret_cast<float4*>(r0) = make_float4(ak[0], ak[1], ak[2], ak[3]);
    *reinterpret_cast<float4*>(r0 + DVS) = make_float4(aq[0], aq[1], aq[2], aq[3]);
  }
  consumer_sync();  // (D)
  if (warp < 4 && rsub == 0) {
    float* r0 = red + warp * 2 * DVS + c4 * 4;
    float4 pk = *reinterpret_cast<float4*>(r0), pq = *reinterpret_cast<float4*>(r0 + DVS);
    pk.x += ak[0];
    pk.y += ak[1];
    pk.z += ak[2];
    pk.w += ak[3];
    pq.x += aq[0];
    pq.y += aq[1];
    pq.z += aq[2];
    pq.w += aq[3];
    *reinterpret_cast<float4*>(r0) = pk;
    *reinterpret_cast<float4*>(r0 + DVS) = pq;
  }
  if (consumer_sync_or(timeout)) {  // (E)
    if (tid == 0) atomic_status(p.status, GDN_STATUS_TIMEOUT);
    return;
  }
  // The step goes ahead. Slice 0 of a split head first waits until slice 1 has read the
  // shared metadata and the q / k conv rows (or has exited), then commits them.
  if (NS > 1 && writer) cluster_wait();
  // only now does the conv cache row shift (a call that timed out above has written
  // nothing, the cache included, so retrying it is safe); slice 0 shifts the q / k rows,
  // every slice the v rows of its columns
  if (conv) {
    if (is_q && writer) conv_commit_channel(p, b, slot, qkv_channel<DK, DV>(p, 0, h, ii), bf16);
    if (is_k && writer) conv_commit_channel(p, b, slot, qkv_channel<DK, DV>(p, 1, h, ii), bf16);
    if (is_col) conv_commit_channel(p, b, slot, qkv_channel<DK, DV>(p, 2, h, col0 + tid), bf16);
  }

  // ---- phase 2: residual, write strength, readout, log commit ----------------------
  float oj = 0.0f;
  if (is_col) {
    const int j = tid;
    float rk = red[j];
    rk += red[2 * DVS + j];
    rk += red[4 * DVS + j];
    rk += red[6 * DVS + j];
    float rq = red[DVS + j];
    rq += red[3 * DVS + j];
    rq += red[5 * DVS + j];
    rq += red[7 * DVS + j];
    // the sums ran on the raw vectors; an explicit rounded product keeps every mode
    // (with or without log terms after it) on the same arithmetic
    rk = __fmul_rn(rk, kinv);
    rq = __fmul_rn(rq, qsc);
    for (int e = 0; e < n; ++e) {
      const float u = (ulb == 2) ? bf16_bits_to_float(u16_s[e * DVS + j]) : u_s[e * DVS + j];
      rk = fmaf(ck_s[e], u, rk);
      rq = fmaf(cq_s[e], u, rq);
    }
    const float bj = (fl & GDN_PLAIN_UPDATE) ? beta * vj : beta * (vj - rk);
    oj = fmaf(scal_f[8] * qsc * kinv, bj, rq);
    if (!(EXT && (fl & GDN_OUT_NORM_GATE))) p.o[(static_cast<size_t>(b) * p.H + h) * DV + col0 + j] = oj;
    b_s[j] = bj;
    if (is_append) {
      const float uval = (fl & GDN_KLOG_PRENORM) ? bj * kinv : bj;
      const size_t at = (sh * C + n) * DV + col0 + j;
      if (ulb == 2)
        reinterpret_cast<__nv_bfloat16*>(p.u_log)[at] = __float2bfloat16_rn(uval);
      else
        static_cast<float*>(p.u_log)[at] = uval;
    }
  }
  if (EXT && (fl & GDN_OUT_NORM_GATE)) {
    // KDA output epilogue: o <- o / sqrt(mean(o^2) + eps) * w * sigmoid(g) over the head's
    // dv channels (the column-owning warps hold them; the other lanes add zero). The RMS
    // needs the whole head, so the epilogue is built for unsplit heads only.
    static_assert(NS == 1 || !EXT, "the output epilogue needs the whole head in one CTA");
    const float ss = warp_sum(oj * oj);
    if (lane == 0 && warp < 4) scal_f[12 + warp] = ss;
    consumer_sync();
    if (is_col) {
      const float ms = (scal_f[12] + scal_f[13] + scal_f[14] + scal_f[15]) / static_cast<float>(DV);
      const float w = p.out_norm_w ? __ldg(p.out_norm_w + tid) : 1.0f;
      p.o[(static_cast<size_t>(b) * p.H + h) * DV + tid] = oj * (1.0f / sqrtf(ms + p.out_eps)) * w * sigmoidf_(og);
    }
  }
  if (is_append) {
    if (is_k && writer) {
      const float kval = (fl & GDN_KLOG_PRENORM) ? x : x * kinv;
      const size_t at = (sh * C + n) * DK + ii;
      if (klb == 2)
        reinterpret_cast<__nv_bfloat16*>(p.k_log)[at] = __float2bfloat16_rn(kval);
      else
        reinterpret_cast<float*>(p.k_log)[at] = kval;
    }
    if (tid < dlam && writer) {
      p.lam_log[(sh * C + n) * dlam + tid] = ellp_s[tid];
      p.ell[sh * dlam + tid] = ellp_s[tid];
    }
    if (tid == 0 && writer) p.len[sh] = n + 1;
  } else if (is_merge && writer) {
    if (tid < dlam) p.ell[sh * dlam + tid] = 0.0f;
    if (tid == 0) p.len[sh] = 0;
  }

  // ---- phase 3: write the state (dense) or fold the log into the base (merge) ------
  // S' = D(ell') S + sum_{i<L} (e^{ell' - Lambda_i} K_i) U_i^T + k b^T: the log terms in
  // groups of 8 (zero-padded), then the current token's term, in that order; with L = 0
  // this is the dense arithmetic exactly.
  if (MODE == MODE_DENSE || is_merge) {
    consumer_sync();  // (F) b and the padded tables are in shared memory
    float* out = p.state + sh * static_cast<size_t>(DK * DV) + col0;
    float4* tilew = reinterpret_cast<float4*>(tile);
    const float4 bb = reinterpret_cast<const float4*>(b_s)[c4];
    const int ng = (MODE == MODE_DENSE) ? 0 : (n + 7) / 8;
    for (int g = 0; g < ng; ++g) {
      float4 u[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (ulb == 2) {
          const uint2 raw = reinterpret_cast<const uint2*>(u16_s + (g * 8 + e) * DVS)[c4];
          u[e] = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                             __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
        } else {
          u[e] = reinterpret_cast<const float4*>(u_s + (g * 8 + e) * DVS)[c4];
        }
      }
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        const int r = it * RPI + warp * RPW + rsub;
        if (r < DK) {
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
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            acc.x = fmaf(wv[e], u[e].x, acc.x);
            acc.y = fmaf(wv[e], u[e].y, acc.y);
            acc.z = fmaf(wv[e], u[e].z, acc.z);
            acc.w = fmaf(wv[e], u[e].w, acc.w);
          }
          if (g == ng - 1) {  // the current token's term, then the write-back
            const float kk = k_s[r] * kinv;
            acc.x = fmaf(kk, bb.x, acc.x);
            acc.y = fmaf(kk, bb.y, acc.y);
            acc.z = fmaf(kk, bb.z, acc.z);
            acc.w = fmaf(kk, bb.w, acc.w);
            *reinterpret_cast<float4*>(out + static_cast<size_t>(r) * DV + c4 * 4) = acc;
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
        if (r < DK) {
          const float4 s = tile4[r * VPR + c4];
          const float dc = dec_s[r], kk = k_s[r] * kinv;
          float4 o4;
          o4.x = fmaf(kk, bb.x, dc * s.x);
          o4.y = fmaf(kk, bb.y, dc * s.y);
          o4.z = fmaf(kk, bb.z, dc * s.z);
          o4.w = fmaf(kk, bb.w, dc * s.w);
          *reinterpret_cast<float4*>(out + static_cast<size_t>(r) * DV + c4 * 4) = o4;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------
// launcher of one (DK, DV, NS) shape

constexpr int kMaxDevices = 64;

inline int sm_count(int dev) {
  static std::atomic<int> cache[kMaxDevices];
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// The state pool as a 2-D fp32 tensor map (rows of DV values), boxes of box_rows x box_cols.
cudaError_t encode_state_map(CUtensorMap* map, const float* pool, size_t rows, int DV, int box_cols, int box_rows);

template <int DK, int DV, int NS, int MODE, bool EXT>
cudaError_t launch_decode_one(const DecodeParams& p, cudaStream_t stream) {
  static std::atomic<uint32_t> configured[kMaxDevices];
  const int klb = (p.flags & GDN_KLOG_FP32) ? 4 : 2;
  const int ulb = (p.flags & GDN_ULOG_BF16) ? 2 : 4;
  const Layout L = decode_layout(MODE, DK, DV / NS, p.C, klb, ulb);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  auto* kern = gdn_decode_kernel<DK, DV, NS, MODE, EXT>;
  if (configured[dev].load(std::memory_order_relaxed) < L.total) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total));
    if (err != cudaSuccess) return err;
    // several tile CTAs per SM only fit with the whole L1/shared array as shared memory
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
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
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT_DECODE, L.total);
    if (err != cudaSuccess) return err;
    rc = (static_cast<uint64_t>(L.total) << 32) | static_cast<uint32_t>(per_sm > 0 ? per_sm : 1);
    resident[dev].store(rc, std::memory_order_relaxed);
  }
  DecodeParams q = p;
  q.prefetch_ahead = static_cast<int>(rc & 0xffffffffu) * sm_count(dev);
  TileMap<NS> map{};
  if constexpr (NS > 1) {
    constexpr int NCH = (DK >= 128) ? 4 : 1;
    err = encode_state_map(&map.map, p.state, static_cast<size_t>(p.num_slots) * p.H * DK, DV, DV / NS, DK / NCH);
    if (err != cudaSuccess) return err;
  }
  // programmatic stream serialisation: the kernel orders its own reads (griddep_wait); the
  // slices of a split head form one cluster
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.H * NS));
  cfg.blockDim = dim3(NT_DECODE);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (NS > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = NS;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  err = cudaLaunchKernelEx(&cfg, kern, q, map);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <int DK, int DV, int NS, bool EXT>
cudaError_t launch_decode_modes(int mode, const DecodeParams& p, cudaStream_t stream) {
  switch (mode) {
    case MODE_DENSE: return launch_decode_one<DK, DV, NS, MODE_DENSE, EXT>(p, stream);
    case MODE_APPEND: return launch_decode_one<DK, DV, NS, MODE_APPEND, EXT>(p, stream);
    case MODE_MERGE: return launch_decode_one<DK, DV, NS, MODE_MERGE, EXT>(p, stream);
    case MODE_STEP: return launch_decode_one<DK, DV, NS, MODE_STEP, EXT>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int DK, int DV, int NS>
cudaError_t launch_decode_shape(int mode, const DecodeParams& p, cudaStream_t stream) {
  if (p.flags & (GDN_GATE_KDA | GDN_OUT_NORM_GATE)) {
    if constexpr (NS == 1) return launch_decode_modes<DK, DV, NS, true>(mode, p, stream);
    else return cudaErrorInvalidValue;  // rejected by the ABI before launch
  }
  return launch_decode_modes<DK, DV, NS, false>(mode, p, stream);
}

}  // namespace shaped
}  // namespace gdn
