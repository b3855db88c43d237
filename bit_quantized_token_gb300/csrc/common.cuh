// Device-side building blocks shared by the decode-step kernels (sm_103a).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace llmq {

constexpr int kGroup = 64;           // 4-bit group size along the input dimension
constexpr int kTileRows = 32;        // rows per unit: lane l of a warp owns row l
constexpr int kQ4UnitBytes = 1152;   // 32 rows x 64 codes (1024 B) + 32 x half2(scale, min)
constexpr int kBF16UnitBytes = 1024; // 32 rows x 16 bf16
constexpr int kBF16UnitCols = 16;
constexpr int kCWarps = 8;           // consumer warps per GEMV CTA
constexpr int kChunkUnits = kCWarps; // units per ring slot: one per consumer warp
constexpr int kGemvThreads = (kCWarps + 1) * 32;  // + one producer warp
constexpr int kRLoc = 10;            // row tiles a reduction window may touch
constexpr int kMaxK = 8192;          // widest GEMV input (held in registers in the prologue)
constexpr int kAttnThreads = 128;

// Device status bits (OR-ed into the model's status word).
enum : int { ST_TIMEOUT = 1, ST_NAN = 2, ST_BAD_TOKEN = 4, ST_CTX_FULL = 8, ST_BOUNDS = 16 };

// The checked build (-DLLMQ_CHECKED=1): every computed index into a weight
// stream, a K/V cache row or a partial-sum array is tested against its
// buffer first; one outside sets ST_BOUNDS in the status word and its access
// is skipped (no trap). In the normal build the test compiles away.
#ifndef LLMQ_CHECKED
#define LLMQ_CHECKED 0
#endif
__device__ __forceinline__ bool in_bounds(int* status, bool ok) {
  if (LLMQ_CHECKED && !ok) {
    atomicOr(status, ST_BOUNDS);
    return false;
  }
  return true;
}

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s for any device wait

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch ---------------------------------------
// Code before pdl_wait() may only read data no kernel of the step writes
// (weights). Every kernel triggers its dependents right after its own wait,
// so a dependent's pre-wait code never overlaps kernels older than this one.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- mbarrier + 1-D bulk copy ----------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity. On timeout sets
// ST_TIMEOUT in *status and returns false; never spins forever.
// A failed poll backs off with __nanosleep so that a waiting warp does not
// take issue slots from the warps it shares a scheduler with.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  unsigned ns = 32;
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(status, ST_TIMEOUT);
      return false;
    }
    __nanosleep(ns);
    ns = ns < 256 ? 2 * ns : 256;
  }
  return true;
}
// The same bound for a consumer of a copy ring, without pauses (its data is
// usually under a microsecond away): the clock is read every 64th poll.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, int* status) {
  unsigned long long t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63) {
      const unsigned long long t = globaltimer();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > kWaitLimitNs) {
        atomicOr(status, ST_TIMEOUT);
        return false;
      }
    }
  }
}
// Global -> shared bulk copy completing on `bar` (addresses 16-B aligned,
// bytes a multiple of 16). Weights are read once per step: evict first.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Loads issued as predicated instructions, so a run of them goes out back to
// back; the result is zero when !pred. The "memory" clobber keeps them after
// the barrier that precedes them.
__device__ __forceinline__ float4 ldcg4_if(const float* ptr, bool pred) {
  float4 v;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %5, 0;\n\t"
      "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
      "@p ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];\n\t}"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(ptr), "r"((uint32_t)pred)
      : "memory");
  return v;
}
__device__ __forceinline__ float2 ldcg2_if(const float* ptr, bool pred) {
  float2 v;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %3, 0;\n\t"
      "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\t"
      "@p ld.global.cg.v2.f32 {%0, %1}, [%2];\n\t}"
      : "=f"(v.x), "=f"(v.y)
      : "l"(ptr), "r"((uint32_t)pred)
      : "memory");
  return v;
}
__device__ __forceinline__ float ldcg1_if(const float* ptr, bool pred) {
  float v;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t"
      "mov.b32 %0, 0;\n\t@p ld.global.cg.f32 %0, [%1];\n\t}"
      : "=f"(v)
      : "l"(ptr), "r"((uint32_t)pred)
      : "memory");
  return v;
}
// Same through the read-only path, for data no kernel writes (norm weights).
__device__ __forceinline__ float4 ldnc4_if(const float* ptr, bool pred) {
  float4 v;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %5, 0;\n\t"
      "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
      "@p ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];\n\t}"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(ptr), "r"((uint32_t)pred)
      : "memory");
  return v;
}

// ---- paired fp32 arithmetic (sm_100+ f32x2) --------------------------------
// Operands are packed into 64-bit registers inside the asm block so that the
// register allocator pairs them without extra moves.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, b, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "sub.rn.f32x2 c, a, b;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// ---- stream-K partition of U work units over N CTAs ------------------------
// CTA c owns units [U*c/N, U*(c+1)/N). A row tile rt (units rt*G .. rt*G+G-1)
// has S partial-sum slots; the CTAs that touch it fill slots 0, 1, ... in CTA
// order and the remaining slots stay zero (buffers are zeroed once at create).
// U * N < 2^32 always holds (U < 2^24 units, N <= 256 CTAs), so 32-bit
// unsigned arithmetic is exact.
// 16-byte asynchronous global -> shared copy (both addresses 16-byte aligned);
// cp_async_wait_all waits for every copy this thread issued.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// 4- or 8-byte asynchronous copy (both addresses aligned to the size)
template <int BYTES>
__device__ __forceinline__ void cp_async_small(void* dst, const void* src) {
  static_assert(BYTES == 4 || BYTES == 8, "cp.async.ca copies 4, 8 or 16 bytes");
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)), "l"(src), "n"(BYTES) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Groups of copies: commit closes the thread's copies issued since the last
// commit into one group; wait_group<N> returns once at most the N most recent
// groups are still in flight.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct Part {
  int U, N, G, S;  // units, CTAs, units per row tile, slots per row tile
  __host__ __device__ int begin(int c) const { return static_cast<int>((unsigned)U * (unsigned)c / (unsigned)N); }
  __host__ __device__ int cta_of(int u) const {
    return static_cast<int>(((unsigned)(u + 1) * (unsigned)N - 1u) / (unsigned)U);
  }
  __host__ __device__ int first_cta(int rt) const { return cta_of(rt * G); }
  __host__ __device__ int n_contrib(int rt) const { return cta_of(rt * G + G - 1) - cta_of(rt * G) + 1; }
};

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }
// Same function with the hardware exponential and division (relative error
// a few 1e-7 over the activation range); __fdividef gives the right limit 0
// when exp(-z) overflows.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

}  // namespace llmq
