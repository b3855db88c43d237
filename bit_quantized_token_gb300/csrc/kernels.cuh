// Decode-step kernels for sm_103a.
//
// The step follows the aot-llm page's per-token pipeline (sequence diagram and
// "The static pipeline emitted for every model"): RMSNorm -> q/k/v matvec ->
// RoPE -> attention over the KV cache -> o matvec + residual -> RMSNorm ->
// gate/up -> SwiGLU -> down + residual, then RMSNorm -> logits -> greedy
// choice. Weights are group-64 4-bit codes with fp16 scale/min (llmopt page,
// "packed group-64 W4A16"); activations stay fp32 and weights are dequantised
// on the fly (aot-llm Metal section: "f32 activations and dequantize weights
// on the fly"); K/V are stored bf16 and widened to fp32 in attention (zynfer
// page, stage M4).
//
// GB300 structure, which differs from the pages' Metal kernels:
//   * Every GEMV is one kernel with a producer warp that streams the CTA's
//     contiguous range of weight units into a shared-memory ring with 1-D bulk
//     copies (cp.async.bulk + mbarrier) and eight consumer warps that
//     dequantise from shared memory. The producer starts before the kernel
//     waits on its predecessor (programmatic dependent launch), so weight
//     streaming overlaps the previous kernel.
//   * Work is split stream-K style: U = row_tiles * groups units over N CTAs,
//     each CTA a contiguous range. A row tile touched by several CTAs leaves
//     one partial sum per CTA; the next kernel adds them in slot order while it
//     builds its own input (RMSNorm / residual / SwiGLU are fused there), so no
//     float atomics are used and results are bit-reproducible.
//   * Attention is flash-decoding: (kv_head, split) CTAs, GQA heads of a group
//     share each K/V row, online softmax, and the last CTA of a kv head
//     combines the splits. The q/k RMSNorm, RoPE and the bf16 append of the
//     current position are done in its prologue.
#pragma once
#include "common.cuh"

namespace llmq {

// ============================================================================
// Dequant-GEMV
// ============================================================================

// 4-bit unit layout (1152 B, 32 rows x 64 inputs of one group):
//   bytes [0,1024): 64 x 16 B, index (h*32 + lane): row `lane`, inputs
//     32h + 8k + i (low nibble of byte 4k+i) and 32h + 8k + 4 + i (high nibble);
//   bytes [1024,1152): 32 x half2(scale, min), one per row.
// Each lane reads its own 16-B words: conflict-free shared loads, and every
// warp-wide load of the global stream is 512 contiguous bytes.
__device__ __forceinline__ float q4_unit_dot(const uint8_t* __restrict__ ub, const float* __restrict__ xg,
                                             float xsum, int lane) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(ub + lane * 16);
  const uint4 c1 = *reinterpret_cast<const uint4*>(ub + 512 + lane * 16);
  const __half2 sm = *reinterpret_cast<const __half2*>(ub + 1024 + lane * 4);
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  // Byte b -> float(2^23 + b) by placing b under the exponent of 2^23; the
  // low nibble is that minus (2^23 + 16*hi), and 16*hi is the latter minus
  // 2^23. All subtractions are exact in fp32.
  const float M = 8388608.0f;
  float l0 = 0.f, l1 = 0.f, h0 = 0.f, h1 = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float4 xa = *reinterpret_cast<const float4*>(xg + 8 * w);
    const float4 xb = *reinterpret_cast<const float4*>(xg + 8 * w + 4);
    const uint32_t v = words[w];
    const uint32_t s0 = __byte_perm(v, 0x4B000000u, 0x7650), s1 = __byte_perm(v, 0x4B000000u, 0x7651);
    const uint32_t s2 = __byte_perm(v, 0x4B000000u, 0x7652), s3 = __byte_perm(v, 0x4B000000u, 0x7653);
    const float b0 = __uint_as_float(s0 & 0xFFFFFFF0u), b1 = __uint_as_float(s1 & 0xFFFFFFF0u);
    const float b2 = __uint_as_float(s2 & 0xFFFFFFF0u), b3 = __uint_as_float(s3 & 0xFFFFFFF0u);
    float q0, q1, q2, q3, r0, r1, r2, r3;
    sub2(q0, q1, __uint_as_float(s0), __uint_as_float(s1), b0, b1);
    sub2(q2, q3, __uint_as_float(s2), __uint_as_float(s3), b2, b3);
    sub2(r0, r1, b0, b1, M, M);
    sub2(r2, r3, b2, b3, M, M);
    fma2(l0, l1, q0, q1, xa.x, xa.y);
    fma2(l0, l1, q2, q3, xa.z, xa.w);
    fma2(h0, h1, r0, r1, xb.x, xb.y);
    fma2(h0, h1, r2, r3, xb.z, xb.w);
  }
  const float d = (l0 + l1) + (h0 + h1) * 0.0625f;  // sum_j q_j x_j
  const float2 s = __half22float2(sm);
  // sum_j (s q_j + m) x_j = s * sum q x + m * sum x
  return fmaf(s.x, d, s.y * xsum);
}

// bf16 unit layout (1024 B, 32 rows x 16 inputs): 2 x 32 x 16 B, index
// (k*32 + lane): row `lane`, inputs 8k .. 8k+7.
__device__ __forceinline__ float bf16_unit_dot(const uint8_t* __restrict__ ub, const float* __restrict__ xg,
                                               int lane) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(ub + lane * 16);
  const uint4 c1 = *reinterpret_cast<const uint4*>(ub + 512 + lane * 16);
  const float4 x0 = *reinterpret_cast<const float4*>(xg);
  const float4 x1 = *reinterpret_cast<const float4*>(xg + 4);
  const float4 x2 = *reinterpret_cast<const float4*>(xg + 8);
  const float4 x3 = *reinterpret_cast<const float4*>(xg + 12);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  fma2(a0, a1, __uint_as_float(c0.x << 16), __uint_as_float(c0.x & 0xFFFF0000u), x0.x, x0.y);
  fma2(a2, a3, __uint_as_float(c0.y << 16), __uint_as_float(c0.y & 0xFFFF0000u), x0.z, x0.w);
  fma2(a0, a1, __uint_as_float(c0.z << 16), __uint_as_float(c0.z & 0xFFFF0000u), x1.x, x1.y);
  fma2(a2, a3, __uint_as_float(c0.w << 16), __uint_as_float(c0.w & 0xFFFF0000u), x1.z, x1.w);
  fma2(a0, a1, __uint_as_float(c1.x << 16), __uint_as_float(c1.x & 0xFFFF0000u), x2.x, x2.y);
  fma2(a2, a3, __uint_as_float(c1.y << 16), __uint_as_float(c1.y & 0xFFFF0000u), x2.z, x2.w);
  fma2(a0, a1, __uint_as_float(c1.z << 16), __uint_as_float(c1.z & 0xFFFF0000u), x3.x, x3.y);
  fma2(a2, a3, __uint_as_float(c1.w << 16), __uint_as_float(c1.w & 0xFFFF0000u), x3.z, x3.w);
  return (a0 + a1) + (a2 + a3);
}

// ---- the 4-bit unit dot over byte limbs ------------------------------------
// Exact integer form of the group's dot product: the group's inputs become
// 32-bit fixed point X_j = rint(x_j 2^sh) with 2^sh chosen so the largest
// |x_j| lands in [2^29, 2^30) (a relative rounding of at most 2^-30 of the
// group's largest input, finer than fp32's own spacing for inputs within 2^6
// of it); sum_j q_j X_j is then formed exactly from byte limbs of X with
// dp4a and combined in 64-bit integers, and converted to fp32 once. The
// scale/min affine map follows: s * 2^-sh * sum q X + m * sum x.
// Unit layout as above: word j = 4h + k of lane l holds the codes of
// inputs 8j .. 8j+3 in its low nibbles and 8j+4 .. 8j+7 in its high nibbles.
// xl: the group's limbs, uint4 [4 limbs][4]; uint4 p of limb k is the byte k
// of X for inputs 16p .. 16p+15 in the order (8j..8j+3, 8j+4..8j+7, 8j+8..,
// 8j+12..) with j = 2p. fe = 2^e / 16, xsum = sum of the group's x.
__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ float q4_unit_dot_limbs(const uint8_t* __restrict__ ub, const uint4* __restrict__ xl,
                                                   float fe, float xsum, int lane, uint32_t mlo, uint32_t mhi) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(ub + lane * 16);
  const uint4 c1 = *reinterpret_cast<const uint4*>(ub + 512 + lane * 16);
  const __half2 sm = *reinterpret_cast<const __half2*>(ub + 1024 + lane * 4);
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  uint32_t lo0 = 0, lo1 = 0, lo2 = 0, hi0 = 0, hi1 = 0, hi2 = 0;
  int lo3 = 0, hi3 = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t wa = words[2 * p], wb = words[2 * p + 1];
    const uint32_t la = wa & mlo, ha = wa & mhi, lb = wb & mlo, hb = wb & mhi;  // hi: 16 x code
    const uint4 x0 = xl[p], x1 = xl[4 + p], x2 = xl[8 + p], x3 = xl[12 + p];
    lo0 = dp4a_uu(la, x0.x, lo0); hi0 = dp4a_uu(ha, x0.y, hi0); lo0 = dp4a_uu(lb, x0.z, lo0); hi0 = dp4a_uu(hb, x0.w, hi0);
    lo1 = dp4a_uu(la, x1.x, lo1); hi1 = dp4a_uu(ha, x1.y, hi1); lo1 = dp4a_uu(lb, x1.z, lo1); hi1 = dp4a_uu(hb, x1.w, hi1);
    lo2 = dp4a_uu(la, x2.x, lo2); hi2 = dp4a_uu(ha, x2.y, hi2); lo2 = dp4a_uu(lb, x2.z, lo2); hi2 = dp4a_uu(hb, x2.w, hi2);
    lo3 = dp4a_us(la, x3.x, lo3); hi3 = dp4a_us(ha, x3.y, hi3); lo3 = dp4a_us(lb, x3.z, lo3); hi3 = dp4a_us(hb, x3.w, hi3);
  }
  // 16 x (sum over limb k) per limb, exact in 32 bits; their weighted sum in 64
  const int c0k = (int)(16u * lo0 + hi0), c1k = (int)(16u * lo1 + hi1), c2k = (int)(16u * lo2 + hi2);
  const int c3k = 16 * lo3 + hi3;
  const int t32 = c3k * 256 + c2k;           // |.| < 2^30
  const int u32 = c1k * 256 + c0k;           // < 2^30
  const long long d64 = (long long)t32 * 65536 + u32;  // 16 * sum_j q_j X_j, exact
  const float d = (float)d64;
  const float2 s = __half22float2(sm);
  return fmaf(s.x * fe, d, s.y * xsum);
}

// The GEMV input as the units read it, from float4 i4 of the (normed) input
// in registers: for 4-bit units the limbs, the exponent factor and the sum of
// each group of 64, for bf16 units the fp32 vector. The 16 threads of a
// half-warp hold one group (every one of them calls this, valid or not). The
// limbs of group g take the bytes of its 64 floats: xl may alias xh, the
// group's threads read their inputs before the shuffles that precede the
// stores.
__device__ __forceinline__ void q4_build_group(float4 x, int i4, bool valid, bool bf16, uint4* xl, float* xh, float* fe,
                                             float* xs) {
  if (bf16) {
    if (valid) reinterpret_cast<float4*>(xh)[i4] = x;
    return;
  }
  float mx = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
  float gs = (x.x + x.y) + (x.z + x.w);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    gs += __shfl_xor_sync(0xffffffffu, gs, o);
  }
  // mx = f * 2^E with f in [0.5, 1): X = x * 2^sh, sh = 30 - E, lies in [-2^30, 2^30]
  // (subnormal mx: E from the scaled value; 2^sh as one or two exact powers of two)
  const uint32_t mb = __float_as_uint(mx);
  int E = (int)((mb >> 23) & 0xFF) - 126;
  if ((mb >> 23) == 0) E = (int)((__float_as_uint(mx * 16777216.0f) >> 23) & 0xFF) - 126 - 24;
  const int sh = 30 - E;
  const int sh1 = sh > 126 ? 126 : sh, sh2 = sh - sh1;  // sh2 > 0 only for tiny groups
  const float p1 = __uint_as_float((uint32_t)(sh1 + 127) << 23);
  const float p2 = __uint_as_float((uint32_t)(sh2 + 127) << 23);
  const bool nz = mx > 0.f;
  const int X0 = nz ? __float2int_rn((x.x * p1) * p2) : 0;
  const int X1 = nz ? __float2int_rn((x.y * p1) * p2) : 0;
  const int X2 = nz ? __float2int_rn((x.z * p1) * p2) : 0;
  const int X3 = nz ? __float2int_rn((x.w * p1) * p2) : 0;
  const uint32_t a_lo = __byte_perm(X0, X1, 0x5140), a_hi = __byte_perm(X0, X1, 0x7362);
  const uint32_t b_lo = __byte_perm(X2, X3, 0x5140), b_hi = __byte_perm(X2, X3, 0x7362);
  if (valid) {
    const int g = i4 >> 4, q = i4 & 15;  // group, quad of the group
    uint32_t* w = reinterpret_cast<uint32_t*>(xl + 16 * g);
    w[0 * 16 + q] = __byte_perm(a_lo, b_lo, 0x5410);
    w[1 * 16 + q] = __byte_perm(a_lo, b_lo, 0x7632);
    w[2 * 16 + q] = __byte_perm(a_hi, b_hi, 0x5410);
    w[3 * 16 + q] = __byte_perm(a_hi, b_hi, 0x7632);
    if (q == 0) {
      const int fx = -sh - 4;  // 2^e / 16 with e = -sh
      fe[g] = !nz ? 0.f : (fx >= -126 ? __uint_as_float((uint32_t)(fx + 127) << 23) : ldexpf(1.0f, fx));
      xs[g] = gs;
    }
  }
}


// ---- W4A8: 4-bit weights x int8 activations ---------------------------------
// The GEMV input quantized once to 8-bit blocks of 32 (the Q8_0 scheme: an
// fp16 scale d = fp16(amax / 127), codes clamp(round(x / d), +-127), rounded
// half away from zero, all in fp32), then an integer dot per block. A group
// of 64 inputs is two blocks; everything a unit reads of group g sits in the
// group's 64-float slot: words 0..15 the codes (word q = inputs 4q .. 4q+3,
// one byte each), word 16/17 the blocks' d / 16, word 18 the min term
// d0 * sum(c of block 0) + d1 * sum(c of block 1).
// Same threads and aliasing as q4_build_group (8 threads per block).
__device__ __forceinline__ void q8_build_group(float4 x, int i4, bool valid, float* slots) {
  float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = __half2float(__float2half_rn(amax / 127.0f));
  auto code = [&](float v) {
    const float c = d == 0.0f ? 0.0f : roundf(v / d);
    return (int)fminf(fmaxf(c, -127.0f), 127.0f);
  };
  const int c0 = code(x.x), c1 = code(x.y), c2 = code(x.z), c3 = code(x.w);
  const uint32_t packed = (uint32_t)(c0 & 0xFF) | ((uint32_t)(c1 & 0xFF) << 8) | ((uint32_t)(c2 & 0xFF) << 16) |
                          ((uint32_t)(c3 & 0xFF) << 24);
  int s2 = (c0 + c1) + (c2 + c3);
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  const float mterm = d * (float)s2;                              // this block's d * sum(c), exact
  const float other = __shfl_xor_sync(0xffffffffu, mterm, 8);   // the group's other block
  if (valid) {
    const int g = i4 >> 4, q = i4 & 15;
    uint32_t* w = reinterpret_cast<uint32_t*>(slots + 64 * g);
    w[q] = packed;
    if ((q & 7) == 0) slots[64 * g + 16 + (q >> 3)] = d * 0.0625f;
    if (q == 0) slots[64 * g + 18] = mterm + other;
  }
}

// One unit against a W4A8 group slot: sum over the two blocks of
// d_b * (scale * sum q c + min * sum c). Lane word j of the unit covers inputs
// 8j .. 8j+7 (low nibbles 8j .. 8j+3, high 8j+4 .. 8j+7): block 0 is words
// 0..3, block 1 words 4..7; the high-nibble sums come out 16 x, which the
// stored d / 16 takes back.
__device__ __forceinline__ float q4a8_unit_dot(const uint8_t* __restrict__ ub, const float* __restrict__ slot,
                                               int lane, uint32_t mlo, uint32_t mhi) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(ub + lane * 16);
  const uint4 c1 = *reinterpret_cast<const uint4*>(ub + 512 + lane * 16);
  const __half2 sm = *reinterpret_cast<const __half2*>(ub + 1024 + lane * 4);
  const uint4* xq = reinterpret_cast<const uint4*>(slot);
  const uint4 xa = xq[0], xb = xq[1], xc = xq[2], xd = xq[3];
  const float4 dm = reinterpret_cast<const float4*>(slot)[4];  // d0 / 16, d1 / 16, min term
  int l0 = 0, h0 = 0, l1 = 0, h1 = 0;
  l0 = dp4a_us(c0.x & mlo, xa.x, l0); h0 = dp4a_us(c0.x & mhi, xa.y, h0);
  l0 = dp4a_us(c0.y & mlo, xa.z, l0); h0 = dp4a_us(c0.y & mhi, xa.w, h0);
  l0 = dp4a_us(c0.z & mlo, xb.x, l0); h0 = dp4a_us(c0.z & mhi, xb.y, h0);
  l0 = dp4a_us(c0.w & mlo, xb.z, l0); h0 = dp4a_us(c0.w & mhi, xb.w, h0);
  l1 = dp4a_us(c1.x & mlo, xc.x, l1); h1 = dp4a_us(c1.x & mhi, xc.y, h1);
  l1 = dp4a_us(c1.y & mlo, xc.z, l1); h1 = dp4a_us(c1.y & mhi, xc.w, h1);
  l1 = dp4a_us(c1.z & mlo, xd.x, l1); h1 = dp4a_us(c1.z & mhi, xd.y, h1);
  l1 = dp4a_us(c1.w & mlo, xd.z, l1); h1 = dp4a_us(c1.w & mhi, xd.w, h1);
  const int t0 = 16 * l0 + h0, t1 = 16 * l1 + h1;  // 16 x sum q c per block, exact
  const float2 s = __half22float2(sm);
  return fmaf(s.x, fmaf(dm.x, (float)t0, dm.y * (float)t1), s.y * dm.z);
}

// How a GEMV kernel gets its fp32 input vector (then optional RMSNorm).
enum VecMode : int {
  VEC_PLAIN = 0,       // v = vin (written by an earlier kernel of the step)
  VEC_EMBED_F32 = 1,   // v = embedding row of the current token
  VEC_EMBED_BF16 = 2,
};
// What a GEMV does with a finished output row y.
enum Epi : int {
  EPI_STORE = 0,       // out[r] = y
  EPI_RESID = 1,       // out[r] = resid[r] + y (residual stream)
  EPI_SWIGLU = 2,      // row tile t = 16 gate rows + 16 up rows: out[16t+i] = silu(g_i) * u_i
  EPI_LOGITS = 3,      // out[r] = y, then greedy choice over all rows (max, lowest index)
};

struct GemvParams {
  const uint8_t* units;  // weight unit stream [n_rt][G] units
  int n_rt, G, K, rows;  // row tiles, units per row, K inputs, real rows (<= 32*n_rt)
  int unit_bytes, nslot, ring_bytes;
  Part part;             // partition of the units over the CTAs
  // input
  int vec_mode;
  const float* vin;
  const void* embed;
  const int* tok;
  int vocab;
  float* vstore;         // VEC_EMBED_*: CTA 0 stores the gathered row here
  const float* norm_w;   // RMSNorm weight, or null
  float eps;
  int w4a8;              // 4-bit units on int8 activation blocks (q8_build_group / q4a8_unit_dot)
  // output
  int epi;
  float* out;
  const float* resid;
  float* part_buf;       // [n_rt][part.S][32] partial sums of row tiles split over CTAs
  int* counters;         // [n_rt], zero between launches
  // EPI_LOGITS: greedy choice, token feedback and position advance
  float* cand_v;         // [part.N]
  int* cand_i;
  int* gcounter;         // zero between launches
  int* tok_io;
  int* argmax_out;
  int* hist;
  int* hist_ctr;
  int hist_cap;
  int* pos;
  int* status;
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCWarps * 32) : "memory"); }

// Deterministic sum over the consumer threads (fixed shuffle tree + warp order).
__device__ __forceinline__ float consumer_sum(float v, float* bred) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) bred[warp] = v;
  consumer_sync();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kCWarps; ++w) s += bred[w];
  consumer_sync();
  return s;
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Apply the epilogue to the finished row tile rt (called by a whole warp).
__device__ __forceinline__ void gemv_epilogue(const GemvParams& p, int rt, int lane, float y, float& bv, int& bi,
                                              bool& nan) {
  const int r = rt * 32 + lane;
  if (p.epi == EPI_SWIGLU) {
    const float up = __shfl_down_sync(0xffffffffu, y, 16);
    if (lane < 16) p.out[rt * 16 + lane] = silu(y) * up;
    return;
  }
  if (r >= p.rows) return;
  if (p.epi == EPI_RESID) {
    p.out[r] = __ldcg(p.resid + r) + y;
  } else {
    p.out[r] = y;
    if (p.epi == EPI_LOGITS) {
      if (y != y) nan = true;
      else if (better(y, r, bv, bi)) { bv = y; bi = r; }
    }
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nslot = p.nslot;
  uint8_t* ring = smem;
  float* xh = reinterpret_cast<float*>(smem + p.ring_bytes);          // [K]
  float* nw = xh + p.K;                                                // [K] norm weight
  float* xs = nw + p.K;                                                // [G], group sums
  float* red = xs + ((p.G + 3) & ~3);                                  // [kRLoc][kCWarps][32]
  float* carry = red + kRLoc * kCWarps * 32;                           // [2][32]
  float* bred = carry + 64;                                            // [kCWarps]
  int* flags = reinterpret_cast<int*>(bred + kCWarps);                 // abort, carry rt x2, issued,
  int* ibest = flags + 4;                                              // [kCWarps] + last flags [4]
  float* fbest = reinterpret_cast<float*>(ibest + kCWarps + 4);        // [kCWarps]
  uint64_t* full = reinterpret_cast<uint64_t*>(fbest + kCWarps);       // 16-B aligned
  uint64_t* empty = full + nslot;

  const int c = blockIdx.x;
  const int u0 = p.part.begin(c), u1 = p.part.begin(c + 1);
  const int n_chunks = (u1 - u0 + kChunkUnits - 1) / kChunkUnits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int UB = p.unit_bytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nslot; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCWarps);
    }
    mbar_fence_init();
    flags[0] = 0;
    flags[1] = -1;
    flags[2] = -1;
    flags[3] = 0;
  }
  __syncthreads();
  pdl_trigger();

  if (warp == kCWarps) {
    // ---------------- producer: stream this CTA's weight units ------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int i = 0; i < n_chunks; ++i) {
        const int s = i % nslot;
        if (i >= nslot && !mbar_wait(&empty[s], ((i / nslot) - 1) & 1, p.status)) {
          flags[0] = 1;
          break;
        }
        const int ub = u0 + i * kChunkUnits;
        const int nu = min(kChunkUnits, u1 - ub);
        mbar_expect_tx(&full[s], nu * UB);
        // (checked build: an index outside the stream copies its first units instead)
        const bool okc = in_bounds(p.status, ub + nu <= p.n_rt * p.G);
        bulk_g2s(ring + s * kChunkUnits * UB, p.units + (okc ? (size_t)ub * UB : 0), nu * UB, &full[s], pol);
        flags[3] = i + 1;  // chunks issued
      }
    }
  } else {
    // ---------------- consumers ------------------------------------------
    const int tid = threadIdx.x;
    const int K = p.K;
    uint32_t mlo, mhi;  // the nibble masks of the W4A8 unit dot, held in registers
    asm volatile("mov.b32 %0, 0x0F0F0F0F;" : "=r"(mlo));
    asm volatile("mov.b32 %0, 0xF0F0F0F0;" : "=r"(mhi));
    // weights of the norm do not depend on earlier kernels: load before waiting
    if (p.norm_w)
      for (int i = tid; i < K / 4; i += kCWarps * 32)
        reinterpret_cast<float4*>(nw)[i] = __ldg(reinterpret_cast<const float4*>(p.norm_w) + i);
    for (int i = tid; i < kRLoc * kCWarps * 32; i += kCWarps * 32) red[i] = 0.f;
    pdl_wait();  // the input vector is written by earlier kernels of the step
    // (1) input vector into registers: thread t holds float4s t, t+256, ...
    // (consecutive threads hold consecutive 16-B pieces, so a 64-input group is
    // 16 threads of one half-warp)
    constexpr int MAXV = kMaxK / 4 / (kCWarps * 32);  // float4s per thread
    float4 v[MAXV];
    const int n4 = K / 4;
    if (p.vec_mode == VEC_PLAIN) {
      const float4* src = reinterpret_cast<const float4*>(p.vin);
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int i = tid + j * kCWarps * 32;
        if (i < n4) v[j] = __ldcg(src + i);
      }
    } else {
      int t = *p.tok;
      if (t < 0 || t >= p.vocab) {
        if (tid == 0) atomicOr(p.status, ST_BAD_TOKEN);
        t = 0;
      }
      if (p.vec_mode == VEC_EMBED_F32) {
        const float4* e = reinterpret_cast<const float4*>(static_cast<const float*>(p.embed) + (size_t)t * K);
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
          const int i = tid + j * kCWarps * 32;
          if (i < n4) v[j] = __ldg(e + i);
        }
      } else {
        const uint2* e = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.embed) + (size_t)t * K);
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
          const int i = tid + j * kCWarps * 32;
          if (i < n4) {
            const uint2 u = __ldg(e + i);
            v[j] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                               __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
          }
        }
      }
      if (p.vstore && c == 0)
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
          const int i = tid + j * kCWarps * 32;
          if (i < n4) reinterpret_cast<float4*>(p.vstore)[i] = v[j];
        }
    }
    // (2) RMSNorm: x / sqrt(mean(x^2) + eps) * w, in registers
    if (p.norm_w) {
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < MAXV; ++j)
        if (tid + j * kCWarps * 32 < n4) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
      ss = consumer_sum(ss, bred);
      const float inv = 1.0f / sqrtf(ss / (float)K + p.eps);
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int i = tid + j * kCWarps * 32;
        if (i < n4) {
          const float4 w4 = reinterpret_cast<const float4*>(nw)[i];
          v[j] = make_float4(v[j].x * inv * w4.x, v[j].y * inv * w4.y, v[j].z * inv * w4.z, v[j].w * inv * w4.w);
        }
      }
    }
    // (3) store, and per-group sums (the min term of every group) by
    // shuffles over the 16 threads holding a group
    const bool a8 = !BF16 && p.w4a8 != 0;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int i = tid + j * kCWarps * 32;
      if (j * kCWarps * 32 >= n4) break;  // uniform: no thread has work at this j
      if (a8) {
        q8_build_group(v[j], i, i < n4, xh);
        continue;
      }
      if (i < n4) reinterpret_cast<float4*>(xh)[i] = v[j];
      if (!BF16) {
        float gs = (i < n4) ? (v[j].x + v[j].y) + (v[j].z + v[j].w) : 0.f;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
        if (i < n4 && (lane & 15) == 0) xs[i / 16] = gs;
      }
    }
    consumer_sync();
    // (4) stream the units: chunk i holds units u0+8i .. u0+8i+7, one per warp
    const int G = p.G;
    const int wch = max(1, ((kRLoc - 2) * G + 1) / kChunkUnits);  // chunks per reduction window
    int win_first = 0, win_idx = 0;
    int cur_rt = -1;
    float acc = 0.f;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    bool nan = false;
    int k_rt = (u0 + warp) / G, k_g = (u0 + warp) - k_rt * G;  // (row tile, group) of this warp's unit
    int win_rt0 = u0 / G;
    for (int i = 0; i < n_chunks; ++i) {
      const int s = i % nslot;
      bool ok = (*(volatile int*)&flags[0]) == 0;
      if (ok) {
        ok = mbar_wait(&full[s], (i / nslot) & 1, p.status);
        if (!ok) *(volatile int*)&flags[0] = 1;
      }
      const int k = u0 + i * kChunkUnits + warp;
      if (ok && k < u1) {
        const int rt = k_rt, g = k_g;
        if (rt != cur_rt) {
          if (cur_rt >= 0) red[((cur_rt - win_rt0) * kCWarps + warp) * 32 + lane] = acc;
          acc = 0.f;
          cur_rt = rt;
        }
        const uint8_t* ub = ring + (s * kChunkUnits + warp) * UB;
        if (BF16) acc += bf16_unit_dot(ub, xh + g * kBF16UnitCols, lane);
        else if (a8) acc += q4a8_unit_dot(ub, xh + g * 64, lane, mlo, mhi);
        else acc += q4_unit_dot(ub, xh + g * 64, xs[g], lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      k_g += kChunkUnits;
      while (k_g >= G) {
        k_g -= G;
        ++k_rt;
      }
      if (i + 1 == n_chunks || i + 1 - win_first == wch) {
        // ---- close the reduction window: sum warps in order; finished rows
        // go through the epilogue, rows shared with other CTAs leave a partial
        if (cur_rt >= 0) red[((cur_rt - win_rt0) * kCWarps + warp) * 32 + lane] = acc;
        acc = 0.f;
        cur_rt = -1;
        consumer_sync();
        const int wu0 = u0 + win_first * kChunkUnits;
        const int wu1 = min(u1, u0 + (i + 1) * kChunkUnits);
        const int rt_a = wu0 / G, rt_b = (wu1 - 1) / G;
        const int next_rt = (wu1 < u1) ? wu1 / G : -1;
        const int carry_in_rt = flags[1 + ((win_idx + 1) & 1)];
        float* cin = carry + ((win_idx + 1) & 1) * 32;
        float* cout = carry + (win_idx & 1) * 32;
        for (int r = rt_a + warp; r <= rt_b; r += kCWarps) {
          const int li = r - rt_a;
          float sum = (r == carry_in_rt) ? cin[lane] : 0.f;
#pragma unroll
          for (int w2 = 0; w2 < kCWarps; ++w2) {
            sum += red[(li * kCWarps + w2) * 32 + lane];
            red[(li * kCWarps + w2) * 32 + lane] = 0.f;
          }
          if (r == next_rt) {
            cout[lane] = sum;
          } else if (r * G < u0 || (r + 1) * G > u1) {
            if (in_bounds(p.status, r < p.n_rt && c - p.part.first_cta(r) < p.part.S))
              p.part_buf[((size_t)r * p.part.S + (c - p.part.first_cta(r))) * 32 + lane] = sum;
          } else {
            gemv_epilogue(p, r, lane, sum, bv, bi, nan);
          }
        }
        if (threadIdx.x == 0) flags[1 + (win_idx & 1)] = (next_rt == rt_b) ? rt_b : -1;
        consumer_sync();
        win_first = i + 1;
        win_rt0 = next_rt;
        ++win_idx;
      }
    }
    // (5) row tiles shared with other CTAs (at most the first and the last):
    // the last CTA to arrive adds the slots in CTA order and runs the epilogue
    const int rt_first = u0 / G, rt_last = (u1 - 1) / G;
    const bool split_first = rt_first * G < u0 || (rt_first + 1) * G > u1;
    const bool split_last = rt_last != rt_first && (rt_last + 1) * G > u1;
    if (split_first || split_last) {
      __threadfence();
      consumer_sync();
      if (threadIdx.x == 0) {
        ibest[kCWarps] = split_first && atomicAdd(&p.counters[rt_first], 1) == p.part.n_contrib(rt_first) - 1;
        ibest[kCWarps + 1] = split_last && atomicAdd(&p.counters[rt_last], 1) == p.part.n_contrib(rt_last) - 1;
      }
      consumer_sync();
      if (warp < 2 && ibest[kCWarps + warp]) {
        __threadfence();
        const int rt = warp == 0 ? rt_first : rt_last;
        const float* src = p.part_buf + (size_t)rt * p.part.S * 32 + lane;
        const int n = p.part.n_contrib(rt);
        float sum = __ldcg(src);
        for (int j = 1; j < n; ++j) sum += __ldcg(src + j * 32);
        gemv_epilogue(p, rt, lane, sum, bv, bi, nan);
        __syncwarp();
        if (lane == 0) p.counters[rt] = 0;
      }
    }
    // (6) logits: greedy choice over all rows, last CTA to arrive decides
    if (p.epi == EPI_LOGITS) {
      if (nan) atomicOr(p.status, ST_NAN);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) { fbest[warp] = bv; ibest[warp] = bi; }
      consumer_sync();
      if (threadIdx.x == 0) {
        for (int w = 0; w < kCWarps; ++w)
          if (better(fbest[w], ibest[w], bv, bi)) { bv = fbest[w]; bi = ibest[w]; }
        p.cand_v[c] = bv;
        p.cand_i[c] = bi;
        __threadfence();
        ibest[kCWarps + 2] = atomicAdd(p.gcounter, 1) == p.part.N - 1;
      }
      consumer_sync();
      if (ibest[kCWarps + 2]) {
        __threadfence();
        bv = -INFINITY;
        bi = 0x7fffffff;
        for (int k = tid; k < p.part.N; k += kCWarps * 32) {
          const float v = __ldcg(p.cand_v + k);
          const int ix = __ldcg(p.cand_i + k);
          if (better(v, ix, bv, bi)) { bv = v; bi = ix; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { fbest[warp] = bv; ibest[warp] = bi; }
        consumer_sync();
        if (threadIdx.x == 0) {
          for (int w = 0; w < kCWarps; ++w)
            if (better(fbest[w], ibest[w], bv, bi)) { bv = fbest[w]; bi = ibest[w]; }
          if (bi < 0 || bi >= p.rows) bi = 0;  // every logit NaN (status already says so)
          *p.argmax_out = bi;
          *p.tok_io = bi;
          const int h = *p.hist_ctr;
          if (h < p.hist_cap) p.hist[h] = bi;
          *p.hist_ctr = h + 1;
          *p.pos = *p.pos + 1;
          *p.gcounter = 0;
        }
      }
    }
  }
  __syncthreads();
  // After an abort, wait (bounded) for copies still landing in the ring.
  if (flags[0] && threadIdx.x == kCWarps * 32) {
    const int issued = flags[3];
    for (int i = max(0, issued - nslot); i < issued; ++i) {  // last chunk issued on each slot
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(&full[i % nslot], (i / nslot) & 1) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  }
}

// ============================================================================
// Attention (flash-decoding) with q/k RMSNorm, RoPE and the bf16 KV append
// ============================================================================
struct AttnParams {
  const float* qkv;       // q|k|v of this step (fused GEMV output)
  int q_dim, kv_dim, Hkv, P;
  const float2* rope;     // [cap][hd/2] (cos, sin) of pos * base^(-2i/hd)
  int rope_neox;
  const float* q_norm;    // [hd] or null
  const float* k_norm;
  float eps;
  uint16_t* kc;           // this layer's cache of the sequence: [Hkv][cap][hd]
  uint16_t* vc;
  int cap;
  const int* pos;         // current position of the sequence
  float* part;            // [Hkv][P][GQ][HD + 2]
  int* counter;           // [Hkv], zero between launches
  float* out;             // [Hq * hd]
  int* status;
};

constexpr int kMinPosPerSplit = 64;

// Number of splits of the cache of length `len` (at most P).
__device__ __forceinline__ int attn_splits(int len, int P) {
  return min(P, max(1, (len + kMinPosPerSplit - 1) / kMinPosPerSplit));
}

// Shared memory of one attention work item.
template <int GQ, int HD, int NW>
struct AttnSmem {
  float qs[GQ][HD];          // scaled query (log2 domain)
  float kv_cur[2][HD];       // current k (rotated) and v, as bf16 values
  float wpart[NW][GQ][HD + 2];
  int is_last;
};

// One (kv head g, split) item of flash-decoding attention, run by NW warps
// that synchronise with Sync::sync(). Reads q|k|v through `load(row)`.
template <int GQ, int HD, int NW, class Sync, class Load>
__device__ void attention_item(const AttnParams& p, int g, int split, int P_eff, int pos, AttnSmem<GQ, HD, NW>& sm,
                               Load load) {
  constexpr int NT = NW * 32;
  constexpr int DPL = HD / 32;  // dims per lane in the V accumulation
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = pos + 1;
  const int t0 = (int)((int64_t)len * split / P_eff), t1 = (int)((int64_t)len * (split + 1) / P_eff);

  // ---- q (GQ heads), k and v of this kv head
  for (int i = tid; i < GQ * HD; i += NT) sm.qs[i / HD][i % HD] = load((g * GQ) * HD + i);
  for (int i = tid; i < 2 * HD; i += NT) {
    const int row = (i < HD) ? (p.q_dim + g * HD + i) : (p.q_dim + p.kv_dim + g * HD + (i - HD));
    sm.kv_cur[i / HD][i % HD] = load(row);
  }
  Sync::sync();
  // ---- per-head RMSNorm of q and k (Qwen3): one warp per head
  if (p.q_norm) {
    for (int h = warp; h <= GQ; h += NW) {
      float* v = (h < GQ) ? sm.qs[h] : sm.kv_cur[0];
      const float* w = (h < GQ) ? p.q_norm : p.k_norm;
      float ss = 0.f;
      for (int d = lane; d < HD; d += 32) ss += v[d] * v[d];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = 1.0f / sqrtf(ss / (float)HD + p.eps);
      __syncwarp();
      for (int d = lane; d < HD; d += 32) v[d] = v[d] * inv * w[d];
    }
    Sync::sync();
  }
  // ---- RoPE at `pos`: pairs (2i, 2i+1) or (i, i + HD/2)
  {
    const float2* cs = p.rope + (size_t)pos * (HD / 2);
    for (int j = tid; j < (GQ + 1) * (HD / 2); j += NT) {
      const int h = j / (HD / 2), i = j % (HD / 2);
      float* v = (h < GQ) ? sm.qs[h] : sm.kv_cur[0];
      const int a = p.rope_neox ? i : 2 * i, b = p.rope_neox ? i + HD / 2 : 2 * i + 1;
      const float2 r = cs[i];
      const float x0 = v[a], x1 = v[b];
      v[a] = x0 * r.x - x1 * r.y;
      v[b] = x0 * r.y + x1 * r.x;
    }
  }
  Sync::sync();
  // ---- round k, v to bf16; the split owning `pos` appends them to the cache
  const float qscale = 1.4426950408889634f / sqrtf((float)HD);  // log2(e)/sqrt(hd)
  for (int i = tid; i < 2 * HD; i += NT) {
    const __nv_bfloat16 b = __float2bfloat16_rn(sm.kv_cur[i / HD][i % HD]);
    sm.kv_cur[i / HD][i % HD] = __bfloat162float(b);
    if (split == P_eff - 1) {
      uint16_t* dst = (i < HD ? p.kc : p.vc) + ((size_t)g * p.cap + pos) * HD + (i % HD);
      *dst = __bfloat16_as_ushort(b);
    }
  }
  for (int i = tid; i < GQ * HD; i += NT) sm.qs[i / HD][i % HD] *= qscale;
  Sync::sync();

  // ---- online softmax over this split's positions, 32 per warp iteration
  float m[GQ], l[GQ], acc[GQ][DPL];
#pragma unroll
  for (int h = 0; h < GQ; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
  }
  const uint16_t* kbase = p.kc + (size_t)g * p.cap * HD;
  const uint16_t* vbase = p.vc + (size_t)g * p.cap * HD;
  if (t1 - t0 <= NW * 8) {
    // short split: warp w takes positions t0+w, t0+w+NW, ...; lane l holds
    // dims l+32e of q, k, v; a score is a butterfly sum over the warp
    float qr[GQ][DPL];
#pragma unroll
    for (int h = 0; h < GQ; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e) qr[h][e] = sm.qs[h][lane + 32 * e];
    for (int t = t0 + warp; t < t1; t += NW) {
      float kf[DPL], vf[DPL];
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        if (t == pos) {
          kf[e] = sm.kv_cur[0][lane + 32 * e];
          vf[e] = sm.kv_cur[1][lane + 32 * e];
        } else {
          kf[e] = bf16_bits_to_f32(__ldg(kbase + (size_t)t * HD + lane + 32 * e));
          vf[e] = bf16_bits_to_f32(__ldg(vbase + (size_t)t * HD + lane + 32 * e));
        }
      }
      float sc[GQ];
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        sc[h] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) sc[h] = fmaf(qr[h][e], kf[e], sc[h]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int h = 0; h < GQ; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], o);
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        const float mn = fmaxf(m[h], sc[h]);
        const float corr = exp2f(m[h] - mn);
        const float pj = exp2f(sc[h] - mn);
        l[h] = l[h] * corr + pj;
        m[h] = mn;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(pj, vf[e], acc[h][e] * corr);
      }
    }
  } else
  for (int tb = t0 + warp * 32; tb < t1; tb += NW * 32) {
    const int t = tb + lane;
    const bool valid = t < t1;
    float s[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) s[h] = 0.f;
    if (valid) {
      if (t == pos) {
#pragma unroll 4
        for (int d = 0; d < HD; ++d) {
          const float kd = sm.kv_cur[0][d];
#pragma unroll
          for (int h = 0; h < GQ; ++h) s[h] = fmaf(sm.qs[h][d], kd, s[h]);
        }
      } else {
        // issue a row's loads before using any of them
        const uint4* kr = reinterpret_cast<const uint4*>(kbase + (size_t)t * HD);
        constexpr int KB = (GQ >= 8 ? 4 : 8) < HD / 8 ? (GQ >= 8 ? 4 : 8) : HD / 8;
#pragma unroll
        for (int c0 = 0; c0 < HD / 8; c0 += KB) {
          uint4 u[KB];
#pragma unroll
          for (int c8 = 0; c8 < KB; ++c8) u[c8] = __ldg(kr + c0 + c8);
#pragma unroll
          for (int c8 = 0; c8 < KB; ++c8) {
            const float kf[8] = {__uint_as_float(u[c8].x << 16), __uint_as_float(u[c8].x & 0xFFFF0000u),
                                 __uint_as_float(u[c8].y << 16), __uint_as_float(u[c8].y & 0xFFFF0000u),
                                 __uint_as_float(u[c8].z << 16), __uint_as_float(u[c8].z & 0xFFFF0000u),
                                 __uint_as_float(u[c8].w << 16), __uint_as_float(u[c8].w & 0xFFFF0000u)};
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
              const float4 qa = *reinterpret_cast<const float4*>(&sm.qs[h][(c0 + c8) * 8]);
              const float4 qb = *reinterpret_cast<const float4*>(&sm.qs[h][(c0 + c8) * 8 + 4]);
              s[h] = fmaf(qa.x, kf[0], s[h]);
              s[h] = fmaf(qa.y, kf[1], s[h]);
              s[h] = fmaf(qa.z, kf[2], s[h]);
              s[h] = fmaf(qa.w, kf[3], s[h]);
              s[h] = fmaf(qb.x, kf[4], s[h]);
              s[h] = fmaf(qb.y, kf[5], s[h]);
              s[h] = fmaf(qb.z, kf[6], s[h]);
              s[h] = fmaf(qb.w, kf[7], s[h]);
            }
          }
        }
      }
    }
    float pr[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      float mx = valid ? s[h] : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mn = fmaxf(m[h], mx);
      const float corr = exp2f(m[h] - mn);  // m = -inf first: exp2(-inf) = 0
      pr[h] = valid ? exp2f(s[h] - mn) : 0.f;
      float ps = pr[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[h] = l[h] * corr + ps;
      m[h] = mn;
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[h][e] *= corr;
    }
    const int nv = min(32, t1 - tb);
    // V rows in groups of 8 positions: all loads of a group are in flight together
    for (int j0 = 0; j0 < nv; j0 += 8) {
      float vv[8][DPL];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int tj = tb + j0 + jj;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          if (j0 + jj >= nv) vv[jj][e] = 0.f;
          else if (tj == pos) vv[jj][e] = sm.kv_cur[1][lane + 32 * e];
          else vv[jj][e] = bf16_bits_to_f32(__ldg(vbase + (size_t)tj * HD + lane + 32 * e));
        }
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          const float pj = __shfl_sync(0xffffffffu, pr[h], (j0 + jj) & 31);
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(pj, vv[jj][e], acc[h][e]);
        }
      }
    }
  }
  // ---- combine the warps of this item
#pragma unroll
  for (int h = 0; h < GQ; ++h) {
#pragma unroll
    for (int e = 0; e < DPL; ++e) sm.wpart[warp][h][lane + 32 * e] = acc[h][e];
    if (lane == 0) {
      sm.wpart[warp][h][HD] = m[h];
      sm.wpart[warp][h][HD + 1] = l[h];
    }
  }
  Sync::sync();
  float* gpart = p.part + (((size_t)g * p.P + split) * GQ) * (HD + 2);
  for (int i = tid; i < GQ * HD; i += NT) {
    const int h = i / HD, d = i % HD;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm.wpart[w][h][HD]);
    float L = 0.f, O = 0.f;
    for (int w = 0; w < NW; ++w) {
      const float f = (sm.wpart[w][h][HD] == -INFINITY) ? 0.f : exp2f(sm.wpart[w][h][HD] - M);
      L += sm.wpart[w][h][HD + 1] * f;
      O += sm.wpart[w][h][d] * f;
    }
    if (P_eff == 1) {
      p.out[(g * GQ + h) * HD + d] = O / L;
    } else {
      gpart[h * (HD + 2) + d] = O;
      if (d == 0) {
        gpart[h * (HD + 2) + HD] = M;
        gpart[h * (HD + 2) + HD + 1] = L;
      }
    }
  }
  if (P_eff == 1) {
    Sync::sync();  // wpart is reused by the next item
    return;
  }
  // ---- last split of this kv head combines all splits (no waiting)
  __threadfence();
  Sync::sync();
  if (tid == 0) sm.is_last = (atomicAdd(&p.counter[g], 1) == P_eff - 1);
  Sync::sync();
  if (sm.is_last) {
    __threadfence();
    const float* hp = p.part + ((size_t)g * p.P * GQ) * (HD + 2);
    for (int i = tid; i < GQ * HD; i += NT) {
      const int h = i / HD, d = i % HD;
      float M = -INFINITY;
      for (int sp = 0; sp < P_eff; ++sp) M = fmaxf(M, __ldcg(hp + ((size_t)sp * GQ + h) * (HD + 2) + HD));
      float L = 0.f, O = 0.f;
      for (int sp = 0; sp < P_eff; ++sp) {
        const float* q = hp + ((size_t)sp * GQ + h) * (HD + 2);
        const float f = exp2f(__ldcg(q + HD) - M);
        L += __ldcg(q + HD + 1) * f;
        O += __ldcg(q + d) * f;
      }
      p.out[(g * GQ + h) * HD + d] = O / L;
    }
    if (tid == 0) p.counter[g] = 0;
  }
  Sync::sync();
}

struct CtaSync {
  __device__ static void sync() { __syncthreads(); }
};

template <int GQ, int HD>
__global__ void __launch_bounds__(kAttnThreads) attention_kernel(const AttnParams p) {
  constexpr int NW = kAttnThreads / 32;
  __shared__ __align__(16) AttnSmem<GQ, HD, NW> sm;
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.y, split = blockIdx.x;
  const int pos = *p.pos;
  if (pos < 0 || pos >= p.cap) {
    if (threadIdx.x == 0 && split == 0 && g == 0) atomicOr(p.status, ST_CTX_FULL);
    return;
  }
  const int P_eff = attn_splits(pos + 1, p.P);
  if (split >= P_eff) return;
  attention_item<GQ, HD, NW, CtaSync>(p, g, split, P_eff, pos, sm, [&](int row) { return __ldcg(p.qkv + row); });
}

}  // namespace llmq
