// Sampled next-token choice on the device, launched after the step in the
// same graph when sampling is on (aot-llm page, "Generated binary options":
// temperature with 0 = greedy, top-k, top-p nucleus threshold, RNG seed).
//
// The choice (the plainest reading of those options): keep the top_k largest
// logits, ties to the lower token id; p_j = softmax((l_j - l_max) / T) in that
// order; keep the shortest prefix whose cumulative probability reaches top_p;
// take the first token of the prefix whose cumulative probability exceeds u
// times the prefix's total. The draw u comes from Philox4x32-10 (Salmon,
// Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011)
// with counter (position, sequence, 0, 0) and key (seed low, seed high word):
// u = (x0 >> 8) / 2^24, so a run is reproducible from the seed alone.
//
// One CTA of 1024 threads: an exact radix select of the k-th largest logit
// (4 passes of 8-bit histograms over order-preserving keys held in registers),
// the k candidates gathered in token order, ranked, then one thread does the
// sequential fp32 softmax, nucleus and draw.
#pragma once
#include "common.cuh"

namespace llmq {

constexpr int kSampleMaxK = 64;
constexpr int kSampleThreads = 1024;
constexpr int kSampleKPT = 32;  // logits a thread keeps per batch (a batch: 32768 logits)

struct SampleCfg {      // the options, in device memory (read by the captured graphs)
  float temperature;    // <= 0: greedy, the kernel keeps the step's choice
  float top_p;          // (0, 1]
  int top_k;            // 1 .. kSampleMaxK
  uint32_t seed_lo, seed_hi;
};

struct SampleParams {
  const float* logits;  // [V]
  int V;
  const SampleCfg* cfg;
  int seq;
  const int* pos;       // the position counter after the step: the logits are those of position *pos - 1
  int* tok_io;          // next input token, or null
  int* choice_out;      // the chosen token
  int* hist;            // the step's history entry hist[*hist_ctr - 1] (if below hist_cap), or null
  const int* hist_ctr;
  int hist_cap;
};

// Philox4x32 with 10 rounds: two 32x32 -> 64-bit products a round, key
// bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// Order-preserving key of a float: a larger value has a larger key (-0 as +0).
__device__ __forceinline__ uint32_t sample_key(float x) {
  uint32_t b = __float_as_uint(x);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive prefix sum of one int per thread over the CTA (fixed order).
__device__ __forceinline__ int sample_scan(int v, int* s_warp, int* s_total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive over warps
    if (lane == 31) *s_total = w;
  }
  __syncthreads();
  const int r = x - v + (warp ? s_warp[warp - 1] : 0);
  __syncthreads();  // s_warp is reused by the next scan
  return r;
}

__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleParams p) {
  constexpr int NT = kSampleThreads;
  __shared__ int hist[256];
  __shared__ int s_bin, s_acc, s_total, s_warp[32];
  __shared__ float cv[kSampleMaxK];
  __shared__ int ci[kSampleMaxK];
  __shared__ float sv[kSampleMaxK];
  __shared__ int si[kSampleMaxK];
  pdl_trigger();
  pdl_wait();
  const SampleCfg cfg = *p.cfg;
  if (!(cfg.temperature > 0.f)) return;
  const int tid = threadIdx.x, V = p.V;
  const int k = min(max(cfg.top_k, 1), min(kSampleMaxK, V));

  // ---- the k-th largest key, 8 bits a pass from the top. A thread keeps the
  // keys of a contiguous chunk in registers (one batch of NT * KPT logits;
  // larger vocabularies are walked batch by batch) and adds runs of equal
  // bins to the histogram at once: the logits share their top bytes.
  constexpr int KPT = kSampleKPT;
  const int span = NT * KPT, nbatch = (V + span - 1) / span;
  uint32_t kr[KPT];  // 0: no logit (no real logit has key 0)
  auto load = [&](int b) {
    const int base = b * span + tid * KPT;
#pragma unroll
    for (int e = 0; e < KPT; ++e) kr[e] = base + e < V ? sample_key(__ldcg(p.logits + base + e)) : 0u;
  };
  if (nbatch == 1) load(0);
  uint32_t prefix = 0u, mask = 0u;
  int krem = k, above = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    __syncthreads();
    for (int b = 0; b < nbatch; ++b) {
      if (nbatch > 1) load(b);
      uint32_t run_bin = 0u;
      int run = 0;
#pragma unroll
      for (int e = 0; e < KPT; ++e) {
        const uint32_t key = kr[e];
        if (key != 0u && (key & mask) == prefix) {
          const uint32_t bin = (key >> shift) & 255u;
          if (run > 0 && bin != run_bin) {
            atomicAdd(&hist[run_bin], run);
            run = 0;
          }
          run_bin = bin;
          ++run;
        }
      }
      if (run > 0) atomicAdd(&hist[run_bin], run);
    }
    __syncthreads();
    if (tid < 32) {  // the bin holding the krem-th largest of the keys still in play
      // lane l sums bins 255-8l .. 248-8l; a scan from the top finds the lane,
      // that lane walks its 8 bins
      int part = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) part += hist[255 - 8 * tid - q];
      int incl = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= krem);
      if (tid == __ffs(hit) - 1) {  // the first lane whose running count reaches krem
        int acc = incl - part, b = 255 - 8 * tid;
        for (int q = 0; q < 7; ++q, --b) {
          if (acc + hist[b] >= krem) break;
          acc += hist[b];
        }
        s_bin = b;
        s_acc = acc;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)s_bin << shift;
    mask |= 0xFFu << shift;
    krem -= s_acc;
    above += s_acc;
    __syncthreads();
  }
  // keys above the threshold `prefix` (all of them) and `krem` keys equal to
  // it, the lowest token ids first: gathered in token order (batch, thread,
  // element) with block-wide scans
  int gt_base = 0, eq_base = 0;
  for (int b = 0; b < nbatch; ++b) {
    if (nbatch > 1) load(b);
    int ngt = 0, neq = 0;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      ngt += kr[e] != 0u && kr[e] > prefix;
      neq += kr[e] != 0u && kr[e] == prefix;
    }
    int rgt = gt_base + sample_scan(ngt, s_warp, &s_total);
    const int tot_gt = s_total;
    int req = eq_base + sample_scan(neq, s_warp, &s_total);
    const int tot_eq = s_total;
    const int base = b * span + tid * KPT;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const uint32_t key = kr[e];
      if (key != 0u && key > prefix) {
        cv[rgt] = __ldcg(p.logits + base + e);
        ci[rgt] = base + e;
        ++rgt;
      } else if (key != 0u && key == prefix) {
        if (req < krem) {
          cv[above + req] = __ldcg(p.logits + base + e);
          ci[above + req] = base + e;
        }
        ++req;
      }
    }
    gt_base += tot_gt;
    eq_base += tot_eq;
  }
  __syncthreads();
  // ---- rank the k candidates: value descending, token id ascending
  if (tid < k) {
    const float v = cv[tid];
    const int id = ci[tid];
    int r = 0;
    for (int j = 0; j < k; ++j) r += (cv[j] > v) || (cv[j] == v && ci[j] < id);
    sv[r] = v;
    si[r] = id;
  }
  __syncthreads();
  // ---- softmax at temperature T, nucleus, draw (sequential fp32, one thread)
  if (tid == 0) {
    const float T = cfg.temperature, m = sv[0];
    float e[kSampleMaxK], S = 0.f;
    for (int j = 0; j < k; ++j) {
      e[j] = expf((sv[j] - m) / T);
      S += e[j];
    }
    float c = 0.f;
    int n = k;
    for (int j = 0; j < k; ++j) {
      c += e[j] / S;
      e[j] = c;  // cumulative probability
      if (n == k && c >= cfg.top_p) n = j + 1;
    }
    const int pos = *p.pos - 1;
    const uint4 x = philox4x32_10(make_uint4((uint32_t)pos, (uint32_t)p.seq, 0u, 0u), make_uint2(cfg.seed_lo, cfg.seed_hi));
    const float u = (float)(x.x >> 8) * (1.0f / 16777216.0f);
    const float target = u * e[n - 1];
    int j = 0;
    while (j < n - 1 && !(e[j] > target)) ++j;
    const int tok = si[j];
    *p.choice_out = tok;
    if (p.tok_io) *p.tok_io = tok;
    if (p.hist) {
      const int h = *p.hist_ctr - 1;
      if (h >= 0 && h < p.hist_cap) p.hist[h] = tok;
    }
  }
}

}  // namespace llmq
