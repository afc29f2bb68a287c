// gdn_device.cuh -- device-side helpers: TMA bulk copies, mbarriers with bounded
// waits, element loads for bf16 / fp32 inputs, warp reductions.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {

constexpr int NT = 256;  // threads per CTA (decode: the compute threads)
constexpr int NW = NT / 32;
constexpr int NT_DECODE = NT + 32;  // decode CTA: NW compute warps and one copy-issuing warp

// Upper bound, in SM clock cycles, on any wait for an asynchronous copy
// (about a second at GB300 clocks). A copy that has not landed by then is
// reported with GDN_STATUS_TIMEOUT instead of hanging the GPU.
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Named barrier 1 over the 256 compute threads (the copy-issuing warp never joins it).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// consumer_sync() that also returns the OR of `pred` over the compute threads.
__device__ __forceinline__ bool consumer_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n"
      "  .reg .pred a, b;\n"
      "  setp.ne.u32 a, %1, 0;\n"
      "  bar.red.or.pred b, 1, 256, a;\n"
      "  selp.u32 %0, 1, 0, b;\n"
      "}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0u;
}

// L2 policy for data read exactly once per step (the base/state tiles).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One TMA bulk copy global -> shared (no tensor map: a contiguous byte range) with an
// L2 cache policy. dst, src 16-byte aligned; bytes a multiple of 16. Completion is
// signalled on `bar` through the transaction count.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Ampere-style asynchronous 4-byte copy global -> shared (no register round trip).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// One arrival on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Programmatic dependent launch: let the next launch in the stream schedule its CTAs once
// every CTA of this grid has issued this (or exited) ...
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// ... and wait until the grids this launch depends on have completed and their memory
// operations are visible (returns at once when there is none).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// TMA prefetch of a contiguous byte range into L2 (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of `bar` to complete; gives up after kWaitLimitCycles
// and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t bits) {
  return __uint_as_float(static_cast<uint32_t>(bits) << 16);
}

// Element i of a bf16 or fp32 array, as float.
__device__ __forceinline__ float load_elem(const void* base, size_t i, bool bf16) {
  if (bf16) return bf16_bits_to_float(__ldg(static_cast<const uint16_t*>(base) + i));
  return __ldg(static_cast<const float*>(base) + i);
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ float log_sigmoidf_(float z) {
  return z < 0.0f ? z - log1pf(expf(z)) : -log1pf(expf(-z));
}

__device__ __forceinline__ float siluf_(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void atomic_status(int32_t* status, uint32_t bits) {
  if (status != nullptr && bits != 0u) atomicOr(status, static_cast<int32_t>(bits));
}

// Width-4 causal conv + SiLU of one channel for one request
// ("去掉分母引入卷积": SiLU(x_{t-3} w0 + x_{t-2} w1 + x_{t-1} w2 + x_t w3)). The cache
// row keeps the last three PRE-conv inputs, column 0 oldest; it is only read here
// (conv_commit_channel shifts it once the step is known to go ahead).
__device__ __forceinline__ float conv_silu_channel(const DecodeParams& p, int b, int slot, int c,
                                                   bool bf16) {
  const size_t row = static_cast<size_t>(slot) * p.channels + c;
  const size_t xi = static_cast<size_t>(b) * p.channels + c;
  const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w) + c);
  float x, s0, s1, s2;
  if (bf16) {
    const uint16_t* cs = static_cast<const uint16_t*>(p.conv_pool) + row * 3;
    x = bf16_bits_to_float(__ldg(static_cast<const uint16_t*>(p.mixed) + xi));
    s0 = bf16_bits_to_float(cs[0]);
    s1 = bf16_bits_to_float(cs[1]);
    s2 = bf16_bits_to_float(cs[2]);
  } else {
    const float* cs = static_cast<const float*>(p.conv_pool) + row * 3;
    x = __ldg(static_cast<const float*>(p.mixed) + xi);
    s0 = cs[0];
    s1 = cs[1];
    s2 = cs[2];
  }
  float acc = s0 * w.x;
  acc = fmaf(s1, w.y, acc);
  acc = fmaf(s2, w.z, acc);
  acc = fmaf(x, w.w, acc);
  if (p.conv_b != nullptr) acc += __ldg(p.conv_b + c);
  return siluf_(acc);
}

// Shift one conv cache row: [s0 s1 s2] <- [s1 s2 x_t] (bit-exact for bf16).
__device__ __forceinline__ void conv_commit_channel(const DecodeParams& p, int b, int slot, int c,
                                                    bool bf16) {
  const size_t row = static_cast<size_t>(slot) * p.channels + c;
  const size_t xi = static_cast<size_t>(b) * p.channels + c;
  if (bf16) {
    uint16_t* cs = static_cast<uint16_t*>(p.conv_pool) + row * 3;
    const uint16_t b1 = cs[1], b2 = cs[2];
    const uint16_t xb = __ldg(static_cast<const uint16_t*>(p.mixed) + xi);
    cs[0] = b1;
    cs[1] = b2;
    cs[2] = xb;
  } else {
    float* cs = static_cast<float*>(p.conv_pool) + row * 3;
    const float f1 = cs[1], f2 = cs[2];
    const float xf = __ldg(static_cast<const float*>(p.mixed) + xi);
    cs[0] = f1;
    cs[1] = f2;
    cs[2] = xf;
  }
}

// Input stage shared by every kernel. Thread roles for a head of size D:
// threads [0, D) own q[i] and v[i]; threads [128, 128 + D) own k[i].
// Returns the raw (pre-normalisation) value in *x; v in *vj for q-threads.
__device__ __forceinline__ void load_token(const DecodeParams& p, int b, int h, int slot, int tid,
                                           float* x, float* vj) {
  const int D = p.D;
  const bool bf16 = (p.flags & GDN_QKV_BF16) != 0u;
  const bool is_q = tid < D;
  const bool is_k = tid >= 128 && tid < 128 + D;
  *x = 0.0f;
  *vj = 0.0f;
  if (!is_q && !is_k) return;
  const int i = is_q ? tid : tid - 128;
  if (p.flags & GDN_FUSE_CONV) {
    const int HD = p.H * D;
    if (is_q) {
      *x = conv_silu_channel(p, b, slot, h * D + i, bf16);
      *vj = conv_silu_channel(p, b, slot, 2 * HD + h * D + i, bf16);
    } else {
      *x = conv_silu_channel(p, b, slot, HD + h * D + i, bf16);
    }
  } else {
    const size_t row = (static_cast<size_t>(b) * p.H + h) * D + i;
    if (is_q) {
      *x = load_elem(p.q, row, bf16);
      *vj = load_elem(p.v, row, bf16);
    } else {
      *x = load_elem(p.k, row, bf16);
    }
  }
}

// Commits the conv cache rows of the channels this thread read in load_token.
__device__ __forceinline__ void conv_commit(const DecodeParams& p, int b, int h, int slot,
                                            int tid) {
  const int D = p.D;
  const bool bf16 = (p.flags & GDN_QKV_BF16) != 0u;
  const int HD = p.H * D;
  if (tid < D) {
    conv_commit_channel(p, b, slot, h * D + tid, bf16);
    conv_commit_channel(p, b, slot, 2 * HD + h * D + tid, bf16);
  } else if (tid >= 128 && tid < 128 + D) {
    conv_commit_channel(p, b, slot, HD + h * D + (tid - 128), bf16);
  }
}

}  // namespace gdn
