// Host runtime and C ABI of the decode step (see include/llmq.h).
//
// One model = one weight arena (repacked 4-bit units, bf16 LM-head units),
// canonical embedding, norm weights, a bf16 KV cache per sequence, a RoPE
// table and the step's scratch buffers, all allocated in llm_model_create.
// A batch-1 step is 5 kernels per layer + LM head + logit/argmax reduction,
// launched with programmatic dependent launch and captured once per sequence
// as a CUDA graph whose kernels read the token and position from device
// memory, so the same graph replays for every step.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>
#include <unordered_map>
#include <vector>

#include "kernels.cuh"
#include "step.cuh"
#include "stepll.cuh"
#include "batch.cuh"
#include "sample.cuh"
#include "llmq.h"

using namespace llmq;

namespace {

thread_local std::string g_create_error = "no error";

struct Mat {            // one fused matrix of the weight arena
  size_t off = 0;       // byte offset of its first unit
  int rows = 0, cols = 0, n_rt = 0, G = 0;
  bool bf16 = false;
  int unit_bytes() const { return bf16 ? kBF16UnitBytes : kQ4UnitBytes; }
  size_t bytes() const { return (size_t)n_rt * G * unit_bytes(); }
};

struct GemvPlan {
  Mat m;
  Part part;
  float* part_buf = nullptr;  // partials of row tiles split over CTAs
  int* counters = nullptr;    // arrival counters of those row tiles
  int nslot = 0, ring = 0;
  size_t smem = 0;
};

// One batched GEMV (M tokens): row tiles per CTA, units per chunk, K splits.
struct BPlan {
  Mat m;
  int rtb = 1, kc = 4, ks = 1, n_blocks = 0;
  size_t smem = 0;
};

BPlan plan_bgemv(const Mat& mat, int n_sm) {
  // 256 inputs per chunk (4 four-bit units or 16 bf16 units per row tile);
  // 1, 2 or 4 row tiles per CTA (8 warps = 16-row halves x unit subsets);
  // enough CTAs to fill the GPU once through the K splits (at most kBKsMax:
  // the merging CTA keeps every split's partial of its 4 tokens in flight)
  BPlan p;
  p.m = mat;
  const int epu = mat.bf16 ? kBF16UnitCols : 64;
  p.kc = 256 / epu;
  // more row tiles per CTA only while the row blocks alone fill the GPU; else
  // one row tile per CTA and just enough K splits to fill it once (split-K
  // costs a partial round trip and a merge; at most kBKsMax splits)
  const int max_ks = std::max(1, (mat.G + p.kc - 1) / p.kc);
  p.rtb = 1;
  for (int r : {4, 2})  // bf16 units: at most 2 row tiles (two CTAs of double-buffered 16 KB units per SM)
    if (mat.n_rt % r == 0 && mat.n_rt / r >= n_sm && (!mat.bf16 || r <= 2)) {
      p.rtb = r;
      break;
    }
  p.n_blocks = mat.n_rt / p.rtb;
  // one split more than filling the GPU once for matrices of few row blocks
  // (measured on the 32-sequence step: 5 -> 6 splits for o and down, 2.559 -> 2.515 ms)
  p.ks = std::min({max_ks, kBKsMax, std::max(1, (n_sm + p.n_blocks - 1) / p.n_blocks + (p.n_blocks < 64 ? 1 : 0))});
  p.smem = bgemv_stage_bytes(p.rtb, p.kc, mat.unit_bytes(), epu);
  return p;
}

// Where a named canonical tensor lives inside a fused matrix.
struct Placement {
  int mat;              // index into model->mats
  int kind;             // 0: rows offset, 1: gate rows (interleaved), 2: up rows (interleaved)
  int row0;
};

// Dynamic shared memory of gemv_kernel (layout in the kernel).
size_t gemv_smem(int ring, int K, int G, int nslot) {
  return (size_t)ring + 8 * (size_t)K + 4 * (size_t)((G + 3) & ~3) + 4 * kRLoc * kCWarps * 32 + 4 * 64 +
         4 * kCWarps + 16 + 4 * (kCWarps + 4) + 4 * kCWarps + 16 * (size_t)nslot;
}

// Canonical nibble of element c in row r.
inline uint8_t nib(const uint8_t* codes, int64_t cols, int64_t r, int64_t c) {
  const uint8_t b = codes[r * (cols / 2) + c / 2];
  return (c & 1) ? (b >> 4) : (b & 15);
}

template <typename F>
void parallel_for(int n, F f) {
  const int nt = std::max(1, std::min<int>(n, (int)std::thread::hardware_concurrency()));
  std::vector<std::thread> th;
  for (int t = 0; t < nt; ++t)
    th.emplace_back([=] {
      for (int i = (int)((int64_t)n * t / nt); i < (int)((int64_t)n * (t + 1) / nt); ++i) f(i);
    });
  for (auto& x : th) x.join();
}

// Write canonical rows of a 4-bit tensor into 4-bit units (see q4_unit_dot).
void repack_q4(uint8_t* units, int G, const uint8_t* codes, const uint16_t* scales, const uint16_t* mins,
               int rows, int cols, int kind, int row0) {
  parallel_for(rows, [&](int r) {
    const int fr = kind == 0 ? row0 + r : (r / 16) * 32 + (kind == 2 ? 16 : 0) + (r % 16);
    const int rt = fr / 32, lane = fr % 32;
    for (int g = 0; g < G; ++g) {
      uint8_t* u = units + ((size_t)rt * G + g) * kQ4UnitBytes;
      for (int h = 0; h < 2; ++h)
        for (int k = 0; k < 4; ++k)
          for (int i = 0; i < 4; ++i) {
            const int e = g * 64 + h * 32 + 8 * k + i;
            u[(h * 32 + lane) * 16 + 4 * k + i] =
                (uint8_t)(nib(codes, cols, r, e) | (nib(codes, cols, r, e + 4) << 4));
          }
      std::memcpy(u + 1024 + lane * 4, &scales[(size_t)r * G + g], 2);
      std::memcpy(u + 1024 + lane * 4 + 2, &mins[(size_t)r * G + g], 2);
    }
  });
}

void unpack_q4(const uint8_t* units, int G, uint8_t* codes, uint16_t* scales, uint16_t* mins, int rows, int cols,
               int kind, int row0) {
  parallel_for(rows, [&](int r) {
    const int fr = kind == 0 ? row0 + r : (r / 16) * 32 + (kind == 2 ? 16 : 0) + (r % 16);
    const int rt = fr / 32, lane = fr % 32;
    uint8_t* cr = codes + (size_t)r * (cols / 2);
    for (int g = 0; g < G; ++g) {
      const uint8_t* u = units + ((size_t)rt * G + g) * kQ4UnitBytes;
      for (int h = 0; h < 2; ++h)
        for (int k = 0; k < 4; ++k)
          for (int i = 0; i < 4; ++i) {
            const int e = g * 64 + h * 32 + 8 * k + i;
            const uint8_t b = u[(h * 32 + lane) * 16 + 4 * k + i];
            const uint8_t lo = b & 15, hi = b >> 4;
            cr[e / 2] = (e & 1) ? (uint8_t)((cr[e / 2] & 15) | (lo << 4)) : (uint8_t)((cr[e / 2] & 0xF0) | lo);
            const int e2 = e + 4;
            cr[e2 / 2] = (e2 & 1) ? (uint8_t)((cr[e2 / 2] & 15) | (hi << 4)) : (uint8_t)((cr[e2 / 2] & 0xF0) | hi);
          }
      std::memcpy(&scales[(size_t)r * G + g], u + 1024 + lane * 4, 2);
      std::memcpy(&mins[(size_t)r * G + g], u + 1024 + lane * 4 + 2, 2);
    }
  });
}

// Dense bf16 [rows][cols] -> bf16 units of 16 inputs (see bf16_unit_dot).
void repack_bf16(uint8_t* units, int G, const uint16_t* data, int rows, int cols) {
  parallel_for(rows, [&](int r) {
    const int rt = r / 32, lane = r % 32;
    for (int g = 0; g < G; ++g) {
      uint8_t* u = units + ((size_t)rt * G + g) * kBF16UnitBytes;
      for (int k = 0; k < 2; ++k)
        std::memcpy(u + (k * 32 + lane) * 16, data + (size_t)r * cols + g * kBF16UnitCols + 8 * k, 16);
    }
  });
}

// Stream-K partition of n_rt row tiles x G units over at most n_cta CTAs.
// The slot count S (CTAs that touch one row tile) is padded to 1, 2 or 4 so
// that the consumers of the partials add a tile's slots inside one warp; the
// CTA count shrinks until no tile has more than 4 contributors.
Part make_part(int n_rt, int G, int n_cta) {
  Part p;
  p.U = n_rt * G;
  p.G = G;
  for (int n = std::max(1, std::min(n_cta, p.U));; --n) {
    p.N = n;
    int s = 1;
    for (int rt = 0; rt < n_rt; ++rt) s = std::max(s, p.n_contrib(rt));
    if (s <= 4 || n == 1) {
      p.S = s <= 1 ? 1 : (s <= 2 ? 2 : 4);
      break;
    }
  }
  return p;
}

}  // namespace

struct llm_model {
  llm_config cfg{};
  int device = 0;
  int n_sm = 0, q_dim = 0, kv_dim = 0, gq = 0;
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  std::string err = "no error";
  int poisoned = 0;  // sticky llm_status

  std::vector<Mat> mats;                      // fused matrices in the arena
  std::unordered_map<std::string, Placement> places;
  std::unordered_map<std::string, std::pair<int64_t, int64_t>> shapes;
  uint8_t* d_arena = nullptr;
  size_t arena_bytes = 0;
  void* d_embed = nullptr;                    // canonical embedding (gather)
  bool embed_bf16 = false;
  float* d_norms = nullptr;
  std::vector<size_t> off_attn_norm, off_ffn_norm, off_q_norm, off_k_norm;
  size_t off_final_norm = 0;
  uint16_t* d_k = nullptr;                    // [B][L][Hkv][cap][hd]
  uint16_t* d_v = nullptr;
  bool kv8 = false;                           // LLM_KV_Q8: the grouped int8 cache instead of d_k / d_v
  bool bkv8_ok = false;                       // the batched kernels read and append it
  int8_t* d_k8 = nullptr;                     // codes [B][L][Hkv][cap][hd]
  int8_t* d_v8 = nullptr;
  uint16_t* d_ks = nullptr;                   // fp16 group scales [B][L][Hkv][cap][hd / 32]
  uint16_t* d_vs = nullptr;
  float2* d_rope = nullptr;                   // [cap][hd/2]

  // step plans
  std::vector<GemvPlan> qkv, wo, gu, down;
  GemvPlan lm;
  int attn_P = 1;

  // scratch: split-row-tile partials and counters (one set per GEMV kind),
  // attention split partials, the step's vectors
  float *d_part = nullptr, *d_attn_part = nullptr;
  int* d_cnt = nullptr;                       // [5 GEMV kinds][max n_rt] + attention [Hkv] + greedy [1]
  float *d_qkv = nullptr, *d_obuf = nullptr, *d_abuf = nullptr, *d_xbuf = nullptr, *d_hbuf = nullptr,
        *d_logits = nullptr, *d_cand_v = nullptr;
  int* d_cand_i = nullptr;
  int* d_attn_cnt = nullptr;
  int* d_greedy_cnt = nullptr;
  // batched step (max_batch > 1)
  std::vector<BPlan> bqkv, bwo, bgu, bdown;
  BPlan blm;
  float *d_bss_x = nullptr, *d_bss_h = nullptr;  // batched: per-(row block, token) sums of squares
  float* d_bhid = nullptr;  // [L+1][max_batch][dim] residual after the embedding and each layer (LLM_DEBUG_BATCH_HIDDEN)
  // batched GEMV inputs staged as XL [64][K] (bf16 high parts, remainders)
  uint16_t *d_bx_hl = nullptr, *d_bh_hl = nullptr, *d_bo_hl = nullptr, *d_ba_hl = nullptr;
  float *d_bx = nullptr, *d_bh = nullptr, *d_bqkv = nullptr,
        *d_blogits = nullptr, *d_bpart = nullptr, *d_battn_part = nullptr, *d_bcand_v = nullptr;
  int *d_bcand_i = nullptr, *d_bcnt = nullptr, *d_battn_cnt = nullptr, *d_bgreedy_cnt = nullptr;
  cudaGraphExec_t bgraph = nullptr;
  size_t bsmem_max = 0;
  int bhead_grid = 0;  // > 0: the batched LM head runs as bhead_kernel on this many CTAs
  // persistent step kernel
  bool use_step = false;
  int step_R = 1;                             // input ranges of the persistent step's GEMVs
  int step_fuse_len = 0;                      // cache lengths the step's o-projection builds attend over itself
  float* d_step_ss = nullptr;                 // [phases][4] per-range sums of squares
  bool step_eager = false;
  Phase* d_phases = nullptr;
  int n_phases = 0;
  int* d_step_sync = nullptr;                 // [2]: arrivals, abort
  // dataflow step kernel (stepll.cuh): several steps per launch
  bool use_ll = false;
  int ll_fuse_len = 0;                        // positions it covers (attention inside the o-projection's build)
  LPhase* d_lphases = nullptr;
  int n_lphases = 0;
  uint64_t* d_ll = nullptr;                   // flagged words of every phase
  uint32_t* d_epoch = nullptr;
  int* d_ll_abort = nullptr;
  uint64_t* d_cand = nullptr;
  unsigned long long* d_stamps = nullptr;     // per-phase timestamps of the last profiled launch
  size_t stamps_steps = 0;
  // per-sequence state
  int *d_pos = nullptr, *d_tok = nullptr, *d_argmax = nullptr, *d_hist = nullptr, *d_hist_ctr = nullptr,
      *d_status = nullptr, *d_prompt = nullptr;
  int* d_pf = nullptr;                        // batched prefill: [tok | pos | seq][pf_cap], then [2][kBM] scratch
  SampleCfg* d_samp = nullptr;                // sampling options (temperature 0: greedy)
  bool sampling = false;
  size_t pf_cap = 0;
  int* h_stage = nullptr;                     // pinned staging (slots: kStage*)
  float* h_logits = nullptr;                  // pinned logits of a batch-1 call with host outputs
  size_t h_logits_n = 0;
  std::vector<int> len;
  std::vector<cudaGraphExec_t> graphs;
  int kernels_per_step = 0;
  size_t device_bytes = 0;
  std::vector<void*> allocs;
};

namespace {

int set_err(llm_model* m, int code, const std::string& msg) {
  if (m) m->err = msg;
  else g_create_error = msg;
  return code;
}

int cuda_fail(llm_model* m, cudaError_t e, const char* what) {
  std::string msg = std::string(what) + ": " + cudaGetErrorString(e);
  if (m) {
    m->poisoned = LLM_ERR_CUDA;
    m->err = msg;
  } else {
    g_create_error = msg;
  }
  return LLM_ERR_CUDA;
}

#define CK(call, what)                                  \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(m, e_, what); \
  } while (0)

// llm_debug_fail_alloc: the device allocation (counted from 1) of the models
// created next that reports cudaErrorMemoryAllocation instead of allocating
std::atomic<int> g_fail_alloc{0};

template <typename T>
cudaError_t dalloc(llm_model* m, T** p, size_t bytes) {
  void* q = nullptr;
  int n = g_fail_alloc.load();
  while (n > 0 && !g_fail_alloc.compare_exchange_weak(n, n - 1)) {
  }
  if (n == 1) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(&q, std::max<size_t>(bytes, 16));
  if (e != cudaSuccess) return e;
  m->allocs.push_back(q);
  m->device_bytes += bytes;
  *p = static_cast<T*>(q);
  return cudaSuccess;
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// An NVTX range over one public call (a no-op unless a profiler listens).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// A kernel's dynamic shared memory limit is process-wide state of the
// device, shared by every model and call that launches the same kernel
// instantiation with different sizes: it is only ever raised.
std::mutex g_smem_limit_mu;
template <typename Kern>
cudaError_t raise_smem_limit(Kern kern, size_t bytes) {
  std::lock_guard<std::mutex> lk(g_smem_limit_mu);
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(&a, kern);
  if (e != cudaSuccess) return e;
  if ((size_t)a.maxDynamicSharedSizeBytes >= bytes) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename Kern, typename Params>
cudaError_t launch(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, const Params& prm) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

GemvPlan plan_gemv(const Mat& mat, int n_sm) {
  GemvPlan g;
  g.m = mat;
  g.part = make_part(mat.n_rt, mat.G, n_sm);
  const int slot = kChunkUnits * mat.unit_bytes();
  g.nslot = 8;
  g.ring = g.nslot * slot;
  g.smem = gemv_smem(g.ring, mat.cols, mat.G, g.nslot);
  return g;
}

GemvParams gemv_params(const llm_model* m, const GemvPlan& g) {
  GemvParams p{};
  p.units = m->d_arena + g.m.off;
  p.n_rt = g.m.n_rt;
  p.G = g.m.G;
  p.K = g.m.cols;
  p.unit_bytes = g.m.unit_bytes();
  p.nslot = g.nslot;
  p.ring_bytes = g.ring;
  p.part = g.part;
  p.rows = g.m.rows;
  p.part_buf = g.part_buf;
  p.counters = g.counters;
  p.eps = m->cfg.norm_eps;
  p.w4a8 = (m->cfg.flags & LLM_W4A8) ? 1 : 0;
  p.status = m->d_status;
  p.vocab = m->cfg.vocab;
  return p;
}

cudaError_t launch_gemv(const llm_model* m, const GemvPlan& g, const GemvParams& p, bool pdl) {
  if (g.m.bf16) return launch(gemv_kernel<true>, dim3(g.part.N), dim3(kGemvThreads), g.smem, m->stream, pdl, p);
  return launch(gemv_kernel<false>, dim3(g.part.N), dim3(kGemvThreads), g.smem, m->stream, pdl, p);
}

template <int GQ, int HD>
cudaError_t launch_attn_t(const llm_model* m, const AttnParams& a, bool pdl) {
  return launch(attention_kernel<GQ, HD>, dim3(m->attn_P, m->cfg.n_kv_heads), dim3(kAttnThreads), 0, m->stream, pdl,
                a);
}

cudaError_t launch_attn(const llm_model* m, const AttnParams& a, bool pdl) {
  const int hd = m->cfg.head_dim;
  switch (m->gq * 1000 + hd) {
    case 1064: return launch_attn_t<1, 64>(m, a, pdl);
    case 2064: return launch_attn_t<2, 64>(m, a, pdl);
    case 4064: return launch_attn_t<4, 64>(m, a, pdl);
    case 8064: return launch_attn_t<8, 64>(m, a, pdl);
    case 1128: return launch_attn_t<1, 128>(m, a, pdl);
    case 2128: return launch_attn_t<2, 128>(m, a, pdl);
    case 4128: return launch_attn_t<4, 128>(m, a, pdl);
    case 8128: return launch_attn_t<8, 128>(m, a, pdl);
  }
  return cudaErrorInvalidValue;
}

// Optional per-launch timing of an eager step.
struct Prof {
  std::vector<cudaEvent_t> ev;
  std::vector<llm_kernel_time> rec;
  int64_t kv_len = 0;
  cudaError_t before(cudaStream_t st) {
    cudaEvent_t e;
    cudaError_t r = cudaEventCreate(&e);
    if (r != cudaSuccess) return r;
    ev.push_back(e);
    return cudaEventRecord(e, st);
  }
  cudaError_t after(cudaStream_t st, int kind, int layer, int64_t bytes) {
    cudaError_t r = before(st);
    rec.push_back({kind, layer, bytes, 0.f});
    return r;
  }
};

// The kernels of one batch-1 step, one launcher each (which: 0 q|k|v GEMV,
// 1 attention, 2 o GEMV, 3 gate|up GEMV, 4 down GEMV, 5 LM head + greedy choice).
enum Which { W_QKV = 0, W_ATTN = 1, W_WO = 2, W_GU = 3, W_DOWN = 4, W_LM = 5 };

cudaError_t launch_one(llm_model* m, int seq, int which, int l, bool pdl) {
  const llm_config& c = m->cfg;
  const int L = c.n_layers, d = c.dim;
  switch (which) {
    case W_QKV: {  // q|k|v = Wqkv * rmsnorm(x_l); x_0 = embedding row (stored by CTA 0)
      GemvParams p = gemv_params(m, m->qkv[l]);
      if (l == 0) {
        p.vec_mode = m->embed_bf16 ? VEC_EMBED_BF16 : VEC_EMBED_F32;
        p.embed = m->d_embed;
        p.tok = m->d_tok + seq;
        p.vstore = m->d_xbuf;
      } else {
        p.vec_mode = VEC_PLAIN;
        p.vin = m->d_xbuf + (size_t)l * d;
      }
      p.norm_w = m->d_norms + m->off_attn_norm[l];
      p.epi = EPI_STORE;
      p.out = m->d_qkv;
      return launch_gemv(m, m->qkv[l], p, pdl);
    }
    case W_ATTN: {  // attention over the cache (+ q/k norm, RoPE, bf16 append)
      AttnParams a{};
      a.qkv = m->d_qkv;
      a.q_dim = m->q_dim;
      a.kv_dim = m->kv_dim;
      a.Hkv = c.n_kv_heads;
      a.P = m->attn_P;
      a.rope = m->d_rope;
      a.rope_neox = c.rope_neox;
      a.q_norm = c.qk_norm ? m->d_norms + m->off_q_norm[l] : nullptr;
      a.k_norm = c.qk_norm ? m->d_norms + m->off_k_norm[l] : nullptr;
      a.eps = c.norm_eps;
      const size_t kvoff = ((size_t)seq * L + l) * (size_t)c.n_kv_heads * c.max_seq * c.head_dim;
      a.kc = m->d_k + kvoff;
      a.vc = m->d_v + kvoff;
      a.cap = c.max_seq;
      a.pos = m->d_pos + seq;
      a.part = m->d_attn_part;
      a.counter = m->d_attn_cnt;
      a.out = m->d_obuf;
      a.status = m->d_status;
      return launch_attn(m, a, pdl);
    }
    case W_WO: {  // h_l = x_l + Wo o
      GemvParams p = gemv_params(m, m->wo[l]);
      p.vec_mode = VEC_PLAIN;
      p.vin = m->d_obuf;
      p.epi = EPI_RESID;
      p.resid = m->d_xbuf + (size_t)l * d;
      p.out = m->d_hbuf + (size_t)l * d;
      return launch_gemv(m, m->wo[l], p, pdl);
    }
    case W_GU: {  // a = silu(Wg rmsnorm(h_l)) * (Wu rmsnorm(h_l))
      GemvParams p = gemv_params(m, m->gu[l]);
      p.vec_mode = VEC_PLAIN;
      p.vin = m->d_hbuf + (size_t)l * d;
      p.norm_w = m->d_norms + m->off_ffn_norm[l];
      p.epi = EPI_SWIGLU;
      p.out = m->d_abuf;
      return launch_gemv(m, m->gu[l], p, pdl);
    }
    case W_DOWN: {  // x_{l+1} = h_l + Wd a
      GemvParams p = gemv_params(m, m->down[l]);
      p.vec_mode = VEC_PLAIN;
      p.vin = m->d_abuf;
      p.epi = EPI_RESID;
      p.resid = m->d_hbuf + (size_t)l * d;
      p.out = m->d_xbuf + (size_t)(l + 1) * d;
      return launch_gemv(m, m->down[l], p, pdl);
    }
    default: {  // logits = W_lm rmsnorm(x_L); greedy choice, token feedback, position += 1
      GemvParams p = gemv_params(m, m->lm);
      p.vec_mode = VEC_PLAIN;
      p.vin = m->d_xbuf + (size_t)L * d;
      p.norm_w = m->d_norms + m->off_final_norm;
      p.epi = EPI_LOGITS;
      p.out = m->d_logits;
      p.cand_v = m->d_cand_v;
      p.cand_i = m->d_cand_i;
      p.gcounter = m->d_greedy_cnt;
      p.tok_io = m->d_tok + seq;
      p.argmax_out = m->d_argmax + seq;
      p.hist = m->d_hist;
      p.hist_ctr = m->d_hist_ctr;
      p.hist_cap = c.max_seq;
      p.pos = m->d_pos + seq;
      return launch_gemv(m, m->lm, p, pdl);
    }
  }
}

// Algorithmic HBM bytes of one launch: weight units, or K/V rows read.
int64_t launch_bytes(const llm_model* m, int which, int l, int64_t kv_len) {
  switch (which) {
    case W_QKV: return (int64_t)m->qkv[l].m.bytes();
    case W_ATTN: return (int64_t)2 * m->cfg.n_kv_heads * kv_len * m->cfg.head_dim * 2;
    case W_WO: return (int64_t)m->wo[l].m.bytes();
    case W_GU: return (int64_t)m->gu[l].m.bytes();
    case W_DOWN: return (int64_t)m->down[l].m.bytes();
    case W_LM: return (int64_t)m->lm.m.bytes();
  }
  return 0;
}

int kind_of(const llm_model* m, int which) {
  if (which == W_ATTN) return 2;
  return (which == W_LM && m->lm.m.bf16) ? 1 : 0;
}

// A cooperative launch of one of the persistent step kernels (all CTAs
// co-resident: their grid barriers and flag waits are safe).
template <typename Params>
cudaError_t launch_cooperative(const llm_model* m, const KernelRef& k, int threads, const Params& prm) {
  if (!k.fn) return cudaErrorInvalidDeviceFunction;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(m->n_sm);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = k.smem;
  cfg.stream = m->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<Params*>(&prm)};
  return cudaLaunchKernelExC(&cfg, k.fn, args);
}

bool step_supported(int gq, int hd) { return (gq == 2 && hd == 64) || (gq == 8 && hd == 64) || (gq == 2 && hd == 128); }

cudaError_t enqueue_persistent_step(llm_model* m, int seq, bool fused, unsigned long long* stamps = nullptr) {
  const llm_config& c = m->cfg;
  StepParams sp{};
  sp.phases = m->d_phases;
  sp.n_phases = m->n_phases;
  sp.R = m->step_R;
  sp.dim = c.dim;
  sp.sync = m->d_step_sync;
  sp.status = m->d_status;
  // the expiry test: a barrier no CTA set can reach, a 1 ms limit
  const bool expire = (c.flags & LLM_TEST_EXPIRE_WAIT) != 0;
  sp.bar_extra = expire ? 1 : 0;
  sp.stamps = stamps;
  sp.wait_ns = expire ? 1000000ull : kWaitLimitNs;
  sp.embed = m->d_embed;
  sp.tok = m->d_tok + seq;
  sp.vocab = c.vocab;
  sp.eps = c.norm_eps;
  sp.q_dim = m->q_dim;
  sp.kv_dim = m->kv_dim;
  sp.Hkv = c.n_kv_heads;
  sp.P = m->attn_P;
  sp.cap = c.max_seq;
  sp.rope_neox = c.rope_neox;
  sp.rope = m->d_rope;
  sp.pos = m->d_pos + seq;
  sp.layer_stride = (size_t)c.n_kv_heads * c.max_seq * c.head_dim;
  const size_t seq_off = (size_t)seq * c.n_layers * sp.layer_stride;
  if (m->kv8) {
    sp.k8_base = m->d_k8 + seq_off;
    sp.v8_base = m->d_v8 + seq_off;
    sp.ks_base = m->d_ks + seq_off / 32;
    sp.vs_base = m->d_vs + seq_off / 32;
  } else {
    sp.k_base = m->d_k + seq_off;
    sp.v_base = m->d_v + seq_off;
  }
  // the split partials of the step kernel share the multi-kernel path's buffer
  sp.attn_o = m->d_attn_part;
  sp.attn_ml = m->d_attn_part + (size_t)c.n_kv_heads * m->attn_P * m->gq * c.head_dim;
  sp.attn_cnt = m->d_attn_cnt;
  sp.obuf = m->d_obuf;
  sp.logits = m->d_logits;
  sp.cand_v = m->d_cand_v;
  sp.cand_i = m->d_cand_i;
  sp.gcounter = m->d_greedy_cnt;
  sp.tok_io = m->d_tok + seq;
  sp.argmax_out = m->d_argmax + seq;
  sp.hist = m->d_hist;
  sp.hist_ctr = m->d_hist_ctr;
  sp.hist_cap = c.max_seq;
  cudaError_t e = cudaMemsetAsync(m->d_step_sync, 0, 2 * sizeof(int), m->stream);
  if (e != cudaSuccess) return e;
  return launch_cooperative(m, step_kernel_ref(m->gq, c.head_dim, fused, (c.flags & LLM_W4A8) != 0, m->kv8), kSThreads,
                            sp);
}


// ---- the dataflow step: n steps of one sequence per cooperative launch
// Steps pos0 .. pos0+n-1 of sequence seq (pos0 = the sequence's device
// position): the input token of step i < n_forced is forced[i] (device), the
// others take the previous step's greedy choice (step 0: d_tok[seq]).
cudaError_t enqueue_ll(llm_model* m, int seq, int n_steps, int n_forced, const int* forced,
                       unsigned long long* stamps = nullptr) {
  const llm_config& c = m->cfg;
  StepLLParams sp{};
  sp.phases = m->d_lphases;
  sp.n_phases = m->n_lphases;
  sp.n_steps = n_steps;
  sp.n_forced = n_forced;
  sp.forced = forced;
  sp.dim = c.dim;
  sp.vocab = c.vocab;
  sp.eps = c.norm_eps;
  sp.epoch = m->d_epoch;
  sp.abort = m->d_ll_abort;
  sp.status = m->d_status;
  sp.embed = m->d_embed;
  sp.q_dim = m->q_dim;
  sp.kv_dim = m->kv_dim;
  sp.Hkv = c.n_kv_heads;
  sp.cap = c.max_seq;
  sp.rope_neox = c.rope_neox;
  sp.rope = m->d_rope;
  sp.pos = m->d_pos + seq;
  sp.layer_stride = (size_t)c.n_kv_heads * c.max_seq * c.head_dim;
  sp.k_base = m->d_k + (size_t)seq * c.n_layers * sp.layer_stride;
  sp.v_base = m->d_v + (size_t)seq * c.n_layers * sp.layer_stride;
  sp.cand = m->d_cand;
  sp.logits = m->d_logits;
  sp.tok_io = m->d_tok + seq;
  sp.argmax_out = m->d_argmax + seq;
  sp.hist = m->d_hist;
  sp.hist_ctr = m->d_hist_ctr;
  sp.hist_cap = c.max_seq;
  sp.stamps = stamps;
  return launch_cooperative(m, stepll_kernel_ref(m->gq, c.head_dim), kLThreads, sp);
}

// Whether steps at positions pos0 .. pos0+n-1 run through the dataflow step.
bool ll_covers(const llm_model* m, int pos0, int n) {
  return m->use_ll && !m->sampling && n > 0 && pos0 + n <= m->ll_fuse_len;
}

// Group blocks per row tile for a phase: the (tile, block) items of the
// CTA with the most tiles spread over the consumer warps with the fewest units
// on the busiest warp (ties: fewer, larger blocks); at most kLRed items.
// A block is at most bs_max units, so that one round of items (one block per
// consumer warp) spans less than the ring minus one slot and every warp works
// on slots the producer can have in flight together.
int ll_blocks(int n_rt, int n_cta, int R, int GR, int bs_max) {
  const int nr = std::max(1, n_cta / R);
  const int nt = (n_rt + nr - 1) / nr;
  int best = 0;
  long best_cost = 0;
  for (int nb = 1; nb <= GR; ++nb) {
    if (GR % nb || (long)nt * nb > kLRed || GR / nb > bs_max) continue;
    const long cost = (((long)nt * nb + kLWarps - 1) / kLWarps) * (GR / nb);
    if (best == 0 || cost < best_cost) {
      best = nb;
      best_cost = cost;
    }
  }
  return best;  // 0: no split fits
}

template <int GQ, int HD>
cudaError_t launch_battn_t(const llm_model* m, const BAttnParams& b, int splits, int rows, bool pdl) {
  const dim3 grid(splits, m->cfg.n_kv_heads, rows);
  if (m->kv8)
    return launch(battn_mma_kernel<GQ, HD, true>, grid, dim3(kBAttnThreads), sizeof(BAttnSmemT<GQ, HD, true>),
                  m->stream, pdl, b);
  return launch(battn_mma_kernel<GQ, HD, false>, grid, dim3(kBAttnThreads), sizeof(BAttnSmemT<GQ, HD, false>),
                m->stream, pdl, b);
}
template <int GQ, int HD>
cudaError_t battn_smem_attr() {
  cudaError_t e = raise_smem_limit(battn_mma_kernel<GQ, HD, false>, sizeof(BAttnSmemT<GQ, HD, false>));
  if (e == cudaSuccess) e = raise_smem_limit(battn_mma_kernel<GQ, HD, true>, sizeof(BAttnSmemT<GQ, HD, true>));
  return e;
}
cudaError_t battn_set_smem(int gq, int hd) {
  switch (gq * 1000 + hd) {
    case 1064: return battn_smem_attr<1, 64>();
    case 2064: return battn_smem_attr<2, 64>();
    case 4064: return battn_smem_attr<4, 64>();
    case 8064: return battn_smem_attr<8, 64>();
    case 1128: return battn_smem_attr<1, 128>();
    case 2128: return battn_smem_attr<2, 128>();
    case 4128: return battn_smem_attr<4, 128>();
    case 8128: return battn_smem_attr<8, 128>();
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_battn(const llm_model* m, const BAttnParams& b, int splits, int rows, bool pdl) {
  switch (m->gq * 1000 + m->cfg.head_dim) {
    case 1064: return launch_battn_t<1, 64>(m, b, splits, rows, pdl);
    case 2064: return launch_battn_t<2, 64>(m, b, splits, rows, pdl);
    case 4064: return launch_battn_t<4, 64>(m, b, splits, rows, pdl);
    case 8064: return launch_battn_t<8, 64>(m, b, splits, rows, pdl);
    case 1128: return launch_battn_t<1, 128>(m, b, splits, rows, pdl);
    case 2128: return launch_battn_t<2, 128>(m, b, splits, rows, pdl);
    case 4128: return launch_battn_t<4, 128>(m, b, splits, rows, pdl);
    case 8128: return launch_battn_t<8, 128>(m, b, splits, rows, pdl);
  }
  return cudaErrorInvalidValue;
}

BGemvParams bgemv_params(const llm_model* m, const BPlan& b, int M) {
  BGemvParams p{};
  p.units = m->d_arena + b.m.off;
  p.n_rt = b.m.n_rt;
  p.G = b.m.G;
  p.K = b.m.cols;
  p.rows = b.m.rows;
  p.bf16 = b.m.bf16;
  p.unit_bytes = b.m.unit_bytes();
  p.epu = b.m.bf16 ? kBF16UnitCols : 64;
  p.M = M;
  p.rtb = b.rtb;
  p.kc = b.kc;
  p.ks = b.ks;
  p.eps = m->cfg.norm_eps;
  p.part = m->d_bpart;
  p.counters = m->d_bcnt;
  p.status = m->d_status;
  return p;
}

cudaError_t launch_bgemv(const llm_model* m, const BPlan& b, const BGemvParams& p, bool pdl) {
  const dim3 grid(b.n_blocks * b.ks);
  if (b.m.bf16) return launch(bgemv_kernel<true>, grid, dim3(kBThreads), b.smem, m->stream, pdl, p);
  return launch(bgemv_kernel<false>, grid, dim3(kBThreads), b.smem, m->stream, pdl, p);
}

// Rows of one pass of the batched pipeline: one token per row.
struct BatchedIO {
  int M;                 // rows (tokens), at most kBM
  const int* tok;        // [M] device tokens
  int* pos;              // [M] device positions (the LM head's greedy epilogue advances them)
  const int* seq;        // [M] cache of each row, or null: row b is sequence b
  bool chunk;            // rows are consecutive tokens of one sequence (a prompt chunk)
  bool lm;               // run the LM head with its greedy choice
  int* tok_io;           // [M] greedy choice fed back as the next token
  int* argmax_out;       // [M]
};

BatchedIO decode_io(llm_model* m) {
  BatchedIO io{};
  io.M = m->cfg.max_batch;
  io.tok = m->d_tok;
  io.pos = m->d_pos;
  io.lm = true;
  io.tok_io = m->d_tok;
  io.argmax_out = m->d_argmax;
  return io;
}

// Enqueue one pass of the batched pipeline on m->stream: a decode step of
// every sequence, or a chunk of a prompt (all rows append their k, v first,
// then attend causally over the cache).
cudaError_t enqueue_batched(llm_model* m, const BatchedIO& io) {
  const llm_config& c = m->cfg;
  const int L = c.n_layers, d = c.dim, B = io.M, F = c.ffn_dim;
  // the hidden-state capture copies sit between the kernels: no programmatic launches then
  const bool capture = m->d_bhid && !io.chunk && io.M == c.max_batch;
  const bool pdl = !(c.flags & LLM_NO_PDL) && !capture;
  auto capture_x = [&](int k) {  // the residual after the embedding (k = 0) or layer k - 1
    return capture ? cudaMemcpyAsync(m->d_bhid + (size_t)k * B * d, m->d_bx, (size_t)B * d * 4,
                                     cudaMemcpyDeviceToDevice, m->stream)
                   : cudaSuccess;
  };
  cudaError_t e;
  BEmbedParams ep{};
  ep.embed = m->d_embed;
  ep.bf16 = m->embed_bf16;
  ep.dim = d;
  ep.vocab = c.vocab;
  ep.M = B;
  ep.tok = io.tok;
  ep.x = m->d_bx;
  ep.ss_out = m->d_bss_x;
  ep.x_hl = m->d_bx_hl;
  ep.norm_w = m->d_norms + m->off_attn_norm[0];
  ep.status = m->d_status;
  if ((e = launch(bembed_kernel, dim3(B), dim3(256), 0, m->stream, false, ep)) != cudaSuccess) return e;
  if ((e = capture_x(0)) != cudaSuccess) return e;
  const size_t kv_layer = (size_t)c.n_kv_heads * c.max_seq * c.head_dim;
  const int qkv_cols = m->q_dim + 2 * m->kv_dim;
  for (int l = 0; l < L; ++l) {
    BGemvParams p = bgemv_params(m, m->bqkv[l], B);  // the input staged with attn_norm[l] applied
    p.xl = m->d_bx_hl;
    p.ss_in = m->d_bss_x;
    p.ss_n = l == 0 ? 1 : m->bdown[l - 1].n_blocks;
    p.epi = EPI_STORE;
    p.out = m->d_bqkv;
    p.out_cols = qkv_cols;
    if ((e = launch_bgemv(m, m->bqkv[l], p, pdl)) != cudaSuccess) return e;
    BAttnParams bp{};
    bp.a.q_dim = m->q_dim;
    bp.a.kv_dim = m->kv_dim;
    bp.a.Hkv = c.n_kv_heads;
    bp.a.P = m->attn_P;
    bp.a.rope = m->d_rope;
    bp.a.rope_neox = c.rope_neox;
    bp.a.q_norm = c.qk_norm ? m->d_norms + m->off_q_norm[l] : nullptr;
    bp.a.k_norm = c.qk_norm ? m->d_norms + m->off_k_norm[l] : nullptr;
    bp.a.eps = c.norm_eps;
    if (m->kv8) {
      bp.k8 = m->d_k8 + (size_t)l * kv_layer;
      bp.v8 = m->d_v8 + (size_t)l * kv_layer;
      bp.ks = m->d_ks + (size_t)l * kv_layer / 32;
      bp.vs = m->d_vs + (size_t)l * kv_layer / 32;
    } else {
      bp.a.kc = m->d_k + (size_t)l * kv_layer;
      bp.a.vc = m->d_v + (size_t)l * kv_layer;
    }
    bp.a.cap = c.max_seq;
    bp.a.part = m->d_battn_part;
    bp.a.counter = m->d_battn_cnt;
    bp.o_hl = m->d_bo_hl;
    bp.a.status = m->d_status;
    bp.qkv = m->d_bqkv;
    bp.qkv_cols = qkv_cols;
    bp.o_cols = m->q_dim;
    bp.pos = io.pos;
    bp.seq = io.seq;
    bp.seq_kv_stride = (size_t)L * kv_layer;
    bp.part_stride = (size_t)c.n_kv_heads * m->attn_P * m->gq * (c.head_dim + 2);
    if (io.chunk) {
      bp.mode = BA_APPEND;
      if ((e = launch_battn(m, bp, 1, B, pdl)) != cudaSuccess) return e;
      bp.mode = BA_ATTEND;
    } else {
      bp.mode = BA_APPEND_ATTEND;
    }
    // splits of LLMQ_BATTN_SPLIT_LEN positions: no cache of this model needs more than its capacity's
    const int splits = std::min(m->attn_P, (c.max_seq + LLMQ_BATTN_SPLIT_LEN - 1) / LLMQ_BATTN_SPLIT_LEN);
    if ((e = launch_battn(m, bp, splits, B, pdl)) != cudaSuccess) return e;
    p = bgemv_params(m, m->bwo[l], B);  // h = x + Wo o (staged for gate|up with ffn_norm[l])
    p.xl = m->d_bo_hl;
    p.epi = EPI_RESID;
    p.resid = m->d_bx;
    p.ss_out = m->d_bss_h;
    p.out = m->d_bh;
    p.out_hl = m->d_bh_hl;
    p.out_norm = m->d_norms + m->off_ffn_norm[l];
    p.out_cols = d;
    if ((e = launch_bgemv(m, m->bwo[l], p, pdl)) != cudaSuccess) return e;
    p = bgemv_params(m, m->bgu[l], B);  // a = silu(Wg rmsnorm(h)) * (Wu rmsnorm(h))
    p.xl = m->d_bh_hl;
    p.ss_in = m->d_bss_h;
    p.ss_n = m->bwo[l].n_blocks;
    p.epi = EPI_SWIGLU;
    p.out_hl = m->d_ba_hl;
    p.out_cols = F;
    if ((e = launch_bgemv(m, m->bgu[l], p, pdl)) != cudaSuccess) return e;
    p = bgemv_params(m, m->bdown[l], B);  // x = h + Wd a (staged with the next RMSNorm applied)
    p.xl = m->d_ba_hl;
    p.epi = EPI_RESID;
    p.resid = m->d_bh;
    p.ss_out = m->d_bss_x;
    p.out = m->d_bx;
    p.out_hl = m->d_bx_hl;
    p.out_norm = m->d_norms + (l + 1 < L ? m->off_attn_norm[l + 1] : m->off_final_norm);
    p.out_cols = d;
    if ((e = launch_bgemv(m, m->bdown[l], p, pdl)) != cudaSuccess) return e;
    if ((e = capture_x(l + 1)) != cudaSuccess) return e;
  }
  if (!io.lm) return cudaSuccess;
  BGemvParams p = bgemv_params(m, m->blm, B);  // logits, greedy choice per sequence, positions += 1
  p.xl = m->d_bx_hl;  // staged with the final norm applied
  p.ss_in = m->d_bss_x;
  p.ss_n = m->bdown[L - 1].n_blocks;
  p.epi = EPI_LOGITS;
  p.out = m->d_blogits;
  p.out_cols = c.vocab;
  p.cand_v = m->d_bcand_v;
  p.cand_i = m->d_bcand_i;
  p.gcounter = m->d_bgreedy_cnt;
  p.tok_io = io.tok_io;
  p.argmax_out = io.argmax_out;
  p.pos = io.pos;
  if (m->bhead_grid)
    return launch(bhead_kernel, dim3(m->bhead_grid), dim3(kHThreads), bhead_smem_bytes(p.K), m->stream, pdl, p);
  return launch_bgemv(m, m->blm, p, pdl);
}

// Enqueue one batch-1 decode step of sequence `seq` on m->stream.
// The sampled choice of sequence seq from `logits` (after the step that wrote them).
cudaError_t launch_sample(llm_model* m, int seq, const float* logits, const int* pos, int* tok_io, int* choice,
                          bool hist) {
  SampleParams sp{};
  sp.logits = logits;
  sp.V = m->cfg.vocab;
  sp.cfg = m->d_samp;
  sp.seq = seq;
  sp.pos = pos;
  sp.tok_io = tok_io;
  sp.choice_out = choice;
  sp.hist = hist ? m->d_hist : nullptr;
  sp.hist_ctr = m->d_hist_ctr;
  sp.hist_cap = m->cfg.max_seq;
  return launch(sample_kernel, dim3(1), dim3(kSampleThreads), 0, m->stream, false, sp);
}

cudaError_t enqueue_step_only(llm_model* m, int seq, Prof* prof, bool fused);

cudaError_t enqueue_step(llm_model* m, int seq, Prof* prof = nullptr, bool fused = false) {
  cudaError_t e = enqueue_step_only(m, seq, prof, fused);
  if (e != cudaSuccess || !m->sampling || prof) return e;
  return launch_sample(m, seq, m->d_logits, m->d_pos + seq, m->d_tok + seq, m->d_argmax + seq, true);
}

cudaError_t enqueue_step_only(llm_model* m, int seq, Prof* prof, bool fused) {
  if (m->use_step && !prof) return enqueue_persistent_step(m, seq, fused);
  const int L = m->cfg.n_layers;
  const bool pdl = !(m->cfg.flags & LLM_NO_PDL) && !prof;
  cudaError_t e;
  auto one = [&](int which, int l, bool use_pdl) -> cudaError_t {
    if (prof && (e = prof->before(m->stream)) != cudaSuccess) return e;
    if ((e = launch_one(m, seq, which, l, use_pdl)) != cudaSuccess) return e;
    if (prof) return prof->after(m->stream, kind_of(m, which), which >= W_LM ? -1 : l,
                                 launch_bytes(m, which, l, prof->kv_len));
    return cudaSuccess;
  };
  for (int l = 0; l < L; ++l) {
    // the first kernel of a step follows host-side copies: no programmatic edge
    if ((e = one(W_QKV, l, pdl && l > 0)) != cudaSuccess) return e;
    for (int which : {W_ATTN, W_WO, W_GU, W_DOWN})
      if ((e = one(which, l, pdl)) != cudaSuccess) return e;
  }
  return one(W_LM, -1, pdl);
}

int status_of(llm_model* m, int st);

int check_status(llm_model* m) {
  if (m->poisoned) return m->poisoned;
  int st = 0;
  CK(cudaMemcpyAsync(&st, m->d_status, sizeof(int), cudaMemcpyDeviceToHost, m->stream), "status read");
  CK(cudaStreamSynchronize(m->stream), "stream sync");
  return status_of(m, st);
}

// The llm_status of a device status word the host has read after a synchronization.
int status_of(llm_model* m, int st) {
  if (m->poisoned) return m->poisoned;
  if (st == 0) return LLM_OK;
  CK(cudaMemsetAsync(m->d_status, 0, sizeof(int), m->stream), "status clear");
  if (st & ST_TIMEOUT) {
    m->poisoned = LLM_ERR_TIMEOUT;
    std::string msg = "a device-side wait exceeded its limit";
    int where = 0;
    if (m->d_ll_abort && cudaMemcpy(&where, m->d_ll_abort, 4, cudaMemcpyDeviceToHost) == cudaSuccess && where > 1) {
      msg += " (flag-synchronised step: CTA " + std::to_string((where - 1) >> 8) + ", wait site " +
             std::to_string((where - 1) & 255);
      // where every CTA was: (step * phases + phase) * 4 + stage (0 build, 1 units, 2 publish)
      std::vector<int> prog(m->n_sm);
      if (cudaMemcpy(prog.data(), m->d_ll_abort + 1, 4 * (size_t)m->n_sm, cudaMemcpyDeviceToHost) == cudaSuccess) {
        std::unordered_map<int, int> hist;
        for (int v : prog) hist[v]++;
        msg += "; CTAs at (phase.stage):";
        for (auto& kv : hist)
          msg += " " + std::to_string(kv.first / 4 % std::max(1, m->n_lphases)) + "." + std::to_string(kv.first % 4) +
                 "x" + std::to_string(kv.second);
      }
      msg += ")";
    }
    return set_err(m, LLM_ERR_TIMEOUT, msg);
  }
  if (st & ST_BOUNDS) {
    m->poisoned = LLM_ERR_CUDA;
    return set_err(m, LLM_ERR_CUDA, "an index left its buffer (checked build)");
  }
  if (st & ST_NAN) return set_err(m, LLM_ERR_NAN, "NaN in the logits");
  if (st & ST_CTX_FULL) return set_err(m, LLM_ERR_CTX_FULL, "position reached max_seq on the device");
  return set_err(m, LLM_ERR_INVALID_ARG, "token id out of range on the device");
}

// One step of sequence seq for the token at position `pos` (known on the
// host: it picks the persistent step's variant for that cache length).
int run_step(llm_model* m, int seq, int pos) {
  const bool fused = m->use_step && pos + 1 <= m->step_fuse_len;
  const bool graph = !(m->cfg.flags & LLM_NO_GRAPH);
  if (!graph || m->step_eager) {  // (the persistent step is two operations: launch them directly)
    CK(enqueue_step(m, seq, nullptr, fused), "step launch");
    return LLM_OK;
  }
  cudaGraphExec_t& slot = m->graphs[2 * seq + (fused ? 1 : 0)];
  if (!slot) {
    cudaGraph_t g = nullptr;
    CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal), "begin capture");
    cudaError_t e = enqueue_step(m, seq, nullptr, fused);
    cudaError_t e2 = cudaStreamEndCapture(m->stream, &g);
    if (m->use_step && (e != cudaSuccess || e2 != cudaSuccess)) {
      // a cooperative launch that this driver does not capture: run the step eagerly
      cudaGetLastError();
      if (g) cudaGraphDestroy(g);
      m->step_eager = true;
      CK(enqueue_step(m, seq, nullptr, fused), "step launch");
      return LLM_OK;
    }
    if (e != cudaSuccess) return cuda_fail(m, e, "step capture");
    if (e2 != cudaSuccess) return cuda_fail(m, e2, "end capture");
    cudaGraphExec_t ge = nullptr;
    e = cudaGraphInstantiate(&ge, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return cuda_fail(m, e, "graph instantiate");
    slot = ge;
  }
  CK(cudaGraphLaunch(slot, m->stream), "graph launch");
  return LLM_OK;
}

int check_model(llm_model* m, int seq) {
  if (!m) return set_err(nullptr, LLM_ERR_INVALID_ARG, "model is NULL");
  if (m->poisoned) return m->poisoned;
  if (seq < 0 || seq >= m->cfg.max_batch) return set_err(m, LLM_ERR_INVALID_ARG, "seq out of range");
  return LLM_OK;
}

int copy_out(llm_model* m, void* dst, const void* src, size_t bytes, bool* host) {
  if (!dst) return LLM_OK;
  if (!is_device_ptr(dst)) *host = true;
  CK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, m->stream), "output copy");
  return LLM_OK;
}

// Pinned staging slots (ints of h_stage): the batch-1 token in, the status
// word, and up to 32 tokens in and 32 choices out of a batched call.
constexpr int kStageTok = 8, kStageStatus = 10, kStageToks = 128, kStageChoice = 160, kStageInts = 256;

// Whether a call's outputs include host memory: such a call ends with one
// synchronization, so its small transfers can go through the pinned slots.
bool host_outputs(const void* a, const void* b) {
  return (a && !is_device_ptr(a)) || (b && !is_device_ptr(b));
}

// Upload n tokens: through a pinned slot when the call synchronizes before
// it returns (the slot is free again by then), else from the caller's memory.
int upload_tokens(llm_model* m, int32_t* dst, const int32_t* src, int n, bool sync_call, int slot) {
  if (sync_call && n <= 32) {
    std::memcpy(m->h_stage + slot, src, (size_t)n * 4);
    CK(cudaMemcpyAsync(dst, m->h_stage + slot, (size_t)n * 4, cudaMemcpyHostToDevice, m->stream), "token upload");
  } else {
    CK(cudaMemcpyAsync(dst, src, (size_t)n * 4, cudaMemcpyDefault, m->stream), "token upload");
  }
  return LLM_OK;
}

// The end of a decode call: device outputs are copied asynchronously; host
// outputs, with the status word, come back through pinned memory after one
// synchronization (large ones directly). Returns the call's llm_status.
int finish_call(llm_model* m, float* logits_out, const float* d_logits, size_t n_logits, int32_t* choice_out,
                const int32_t* d_choice, size_t n_choice) {
  const bool hl = logits_out && !is_device_ptr(logits_out);
  const bool hc = choice_out && !is_device_ptr(choice_out);
  if (logits_out && !hl)
    CK(cudaMemcpyAsync(logits_out, d_logits, n_logits * 4, cudaMemcpyDeviceToDevice, m->stream), "output copy");
  if (choice_out && !hc)
    CK(cudaMemcpyAsync(choice_out, d_choice, n_choice * 4, cudaMemcpyDeviceToDevice, m->stream), "output copy");
  if (!hl && !hc) return LLM_OK;  // asynchronous: a later synchronizing call reports the status
  float* lst = (hl && n_logits <= m->h_logits_n) ? m->h_logits : nullptr;
  int32_t* cst = (hc && n_choice <= 32) ? m->h_stage + kStageChoice : nullptr;
  if (hl) CK(cudaMemcpyAsync(lst ? lst : logits_out, d_logits, n_logits * 4, cudaMemcpyDeviceToHost, m->stream),
             "logits copy");
  if (hc) CK(cudaMemcpyAsync(cst ? cst : choice_out, d_choice, n_choice * 4, cudaMemcpyDeviceToHost, m->stream),
             "choice copy");
  CK(cudaMemcpyAsync(m->h_stage + kStageStatus, m->d_status, 4, cudaMemcpyDeviceToHost, m->stream), "status read");
  CK(cudaStreamSynchronize(m->stream), "stream sync");
  if (lst) std::memcpy(logits_out, lst, n_logits * 4);
  if (cst) std::memcpy(choice_out, cst, n_choice * 4);
  return status_of(m, m->h_stage[kStageStatus]);
}

}  // namespace

extern "C" {

const char* llm_last_error(const llm_model* m) { return m ? m->err.c_str() : g_create_error.c_str(); }

void llm_model_destroy(llm_model* m) {
  if (!m) return;
  for (auto g : m->graphs)
    if (g) cudaGraphExecDestroy(g);
  if (m->bgraph) cudaGraphExecDestroy(m->bgraph);
  for (void* p : m->allocs) cudaFree(p);
  if (m->h_stage) cudaFreeHost(m->h_stage);
  if (m->h_logits) cudaFreeHost(m->h_logits);
  if (m->own_stream && m->stream) cudaStreamDestroy(m->stream);
  delete m;
}

int llm_model_create(const llm_config* cfg, const llm_tensor* tensors, int32_t n_tensors, void* cuda_stream,
                     llm_model** out) {
  NvtxRange nvtx_("llm_model_create");
  llm_model* m = nullptr;
  if (out) *out = nullptr;
  if (!cfg || !tensors || !out || n_tensors <= 0)
    return set_err(nullptr, LLM_ERR_INVALID_ARG, "null config, tensors or out pointer");
  if (cfg->abi_version != LLMQ_ABI_VERSION) return set_err(nullptr, LLM_ERR_UNSUPPORTED, "abi_version mismatch");
  const llm_config& c = *cfg;
  if (c.dim <= 0 || c.n_layers <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.ffn_dim <= 0 || c.vocab <= 0 ||
      c.max_seq <= 0 || c.max_batch <= 0 || !(c.norm_eps > 0.f) || !(c.rope_theta > 0.0))
    return set_err(nullptr, LLM_ERR_INVALID_ARG, "non-positive dimension, max_seq, max_batch, eps or theta");
  if (c.head_dim != 64 && c.head_dim != 128)
    return set_err(nullptr, LLM_ERR_UNSUPPORTED, "head_dim=" + std::to_string(c.head_dim) + " (64 or 128 only)");
  if (c.n_heads % c.n_kv_heads)
    return set_err(nullptr, LLM_ERR_UNSUPPORTED, "n_heads not a multiple of n_kv_heads");
  const int gq = c.n_heads / c.n_kv_heads;
  if (gq != 1 && gq != 2 && gq != 4 && gq != 8)
    return set_err(nullptr, LLM_ERR_UNSUPPORTED, "GQA group of " + std::to_string(gq) + " (1, 2, 4 or 8 only)");
  if (c.dim % 64 || c.ffn_dim % 64)
    return set_err(nullptr, LLM_ERR_UNSUPPORTED, "dim and ffn_dim must be multiples of the group size 64");
  if (c.ffn_dim > kMaxK || c.dim > kMaxK || c.n_heads * c.head_dim > kMaxK)
    return set_err(nullptr, LLM_ERR_UNSUPPORTED, "a GEMV input wider than " + std::to_string(kMaxK));
  if (c.rope_neox != 0 && c.rope_neox != 1) return set_err(nullptr, LLM_ERR_INVALID_ARG, "rope_neox must be 0 or 1");
  if (c.max_batch > kBM)
    return set_err(nullptr, LLM_ERR_UNSUPPORTED, "max_batch=" + std::to_string(c.max_batch) + " (32 sequences at most)");

  std::unordered_map<std::string, const llm_tensor*> by_name;
  for (int i = 0; i < n_tensors; ++i)
    if (tensors[i].name) by_name[tensors[i].name] = &tensors[i];
  auto find = [&](const std::string& n, int dtype, int64_t rows, int64_t cols, const llm_tensor** t) -> int {
    auto it = by_name.find(n);
    if (it == by_name.end()) return set_err(nullptr, LLM_ERR_NOT_FOUND, "missing tensor " + n);
    const llm_tensor* x = it->second;
    if (x->dtype != dtype) return set_err(nullptr, LLM_ERR_UNSUPPORTED, "tensor " + n + ": unexpected dtype");
    if (x->rows != rows || x->cols != cols)
      return set_err(nullptr, LLM_ERR_INVALID_ARG,
                     "tensor " + n + ": shape " + std::to_string(x->rows) + "x" + std::to_string(x->cols) +
                         ", expected " + std::to_string(rows) + "x" + std::to_string(cols));
    if (dtype == LLM_Q4G64 ? (!x->codes || !x->scales || !x->mins) : !x->data)
      return set_err(nullptr, LLM_ERR_INVALID_ARG, "tensor " + n + ": null data");
    *t = x;
    return LLM_OK;
  };

  m = new llm_model();
  m->cfg = c;
  m->gq = gq;
  m->q_dim = c.n_heads * c.head_dim;
  m->kv_dim = c.n_kv_heads * c.head_dim;
  int rc;
  auto fail = [&](int code) {
    if (code != LLM_OK && m) {
      if (m->err != "no error") g_create_error = m->err;
      llm_model_destroy(m);
      m = nullptr;
    }
    return code;
  };
  int dev = 0;
  {
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(cuda_fail(nullptr, e, "no CUDA device"));
    m->device = dev;
  }
  const int L = c.n_layers, d = c.dim, F = c.ffn_dim, hd = c.head_dim, V = c.vocab;

  // ---- lay out the arena: per layer QKV, WO, GU, DOWN; then the LM head
  size_t off = 0;
  auto add_mat = [&](int rows, int cols, bool bf16) {
    Mat x;
    x.rows = rows;
    x.cols = cols;
    x.n_rt = (rows + 31) / 32;
    x.G = cols / (bf16 ? kBF16UnitCols : 64);
    x.bf16 = bf16;
    x.off = off;
    off += (x.bytes() + 255) / 256 * 256;
    m->mats.push_back(x);
    return (int)m->mats.size() - 1;
  };
  std::vector<int> mi_qkv(L), mi_wo(L), mi_gu(L), mi_down(L);
  for (int l = 0; l < L; ++l) {
    const std::string P = "L" + std::to_string(l) + ".";
    mi_qkv[l] = add_mat(m->q_dim + 2 * m->kv_dim, d, false);
    m->places[P + "wq"] = {mi_qkv[l], 0, 0};
    m->places[P + "wk"] = {mi_qkv[l], 0, m->q_dim};
    m->places[P + "wv"] = {mi_qkv[l], 0, m->q_dim + m->kv_dim};
    mi_wo[l] = add_mat(d, m->q_dim, false);
    m->places[P + "wo"] = {mi_wo[l], 0, 0};
    mi_gu[l] = add_mat(2 * F, d, false);
    m->places[P + "w_gate"] = {mi_gu[l], 1, 0};
    m->places[P + "w_up"] = {mi_gu[l], 2, 0};
    mi_down[l] = add_mat(d, F, false);
    m->places[P + "w_down"] = {mi_down[l], 0, 0};
    m->shapes[P + "wq"] = {m->q_dim, d};
    m->shapes[P + "wk"] = {m->kv_dim, d};
    m->shapes[P + "wv"] = {m->kv_dim, d};
    m->shapes[P + "wo"] = {d, m->q_dim};
    m->shapes[P + "w_gate"] = {F, d};
    m->shapes[P + "w_up"] = {F, d};
    m->shapes[P + "w_down"] = {d, F};
  }
  const int mi_lm = add_mat(V, d, c.tied_embedding != 0);
  if (!c.tied_embedding) {
    m->places["lm_head"] = {mi_lm, 0, 0};
    m->shapes["lm_head"] = {V, d};
  }
  m->arena_bytes = off;

  // ---- validate inputs and repack on the host
  std::vector<uint8_t> arena(off, 0);
  for (const auto& kv : m->places) {
    const llm_tensor* t = nullptr;
    const auto shp = m->shapes[kv.first];
    if ((rc = find(kv.first, LLM_Q4G64, shp.first, shp.second, &t)) != LLM_OK) return fail(rc);
    const Mat& x = m->mats[kv.second.mat];
    repack_q4(arena.data() + x.off, x.G, static_cast<const uint8_t*>(t->codes), static_cast<const uint16_t*>(t->scales),
              static_cast<const uint16_t*>(t->mins), (int)t->rows, (int)t->cols, kv.second.kind, kv.second.row0);
  }
  const llm_tensor* emb = nullptr;
  m->embed_bf16 = c.tied_embedding != 0;
  if ((rc = find("embed", m->embed_bf16 ? LLM_BF16 : LLM_F32, V, d, &emb)) != LLM_OK) {
    if (rc == LLM_ERR_UNSUPPORTED && c.tied_embedding) g_create_error = "tied embedding must be LLM_BF16";
    return fail(rc);
  }
  if (c.tied_embedding) {
    const Mat& x = m->mats[mi_lm];
    repack_bf16(arena.data() + x.off, x.G, static_cast<const uint16_t*>(emb->data), V, d);
  }
  // norm weights
  std::vector<float> norms;
  auto add_norm = [&](const std::string& n, int len, size_t* where) -> int {
    const llm_tensor* t = nullptr;
    int r = find(n, LLM_F32, 1, len, &t);
    if (r != LLM_OK) return r;
    *where = norms.size();
    const float* src = static_cast<const float*>(t->data);
    norms.insert(norms.end(), src, src + len);
    while (norms.size() % 4) norms.push_back(0.f);
    return LLM_OK;
  };
  m->off_attn_norm.resize(L);
  m->off_ffn_norm.resize(L);
  m->off_q_norm.resize(L);
  m->off_k_norm.resize(L);
  for (int l = 0; l < L; ++l) {
    const std::string P = "L" + std::to_string(l) + ".";
    if ((rc = add_norm(P + "attn_norm", d, &m->off_attn_norm[l])) != LLM_OK) return fail(rc);
    if ((rc = add_norm(P + "ffn_norm", d, &m->off_ffn_norm[l])) != LLM_OK) return fail(rc);
    if (c.qk_norm) {
      if ((rc = add_norm(P + "q_norm", hd, &m->off_q_norm[l])) != LLM_OK) return fail(rc);
      if ((rc = add_norm(P + "k_norm", hd, &m->off_k_norm[l])) != LLM_OK) return fail(rc);
    }
  }
  if ((rc = add_norm("final_norm", d, &m->off_final_norm)) != LLM_OK) return fail(rc);

  // ---- device allocations (all of them, once)
  if (cuda_stream) {
    m->stream = static_cast<cudaStream_t>(cuda_stream);
  } else {
    cudaError_t e = cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return fail(cuda_fail(nullptr, e, "stream create"));
    m->own_stream = true;
  }
  auto A = [&](auto** p, size_t bytes, const char* what) -> int {
    cudaError_t e = dalloc(m, p, bytes);
    if (e == cudaErrorMemoryAllocation) {
      cudaGetLastError();
      return set_err(m, LLM_ERR_OOM, std::string("device allocation failed: ") + what);
    }
    if (e != cudaSuccess) return cuda_fail(m, e, what);
    return LLM_OK;
  };
#define AL(ptr, bytes, what) \
  if ((rc = A(&(ptr), (bytes), (what))) != LLM_OK) return fail(rc)
  AL(m->d_arena, m->arena_bytes, "weights");
  const size_t emb_bytes = (size_t)V * d * (m->embed_bf16 ? 2 : 4);
  AL(m->d_embed, emb_bytes, "embedding");
  AL(m->d_norms, norms.size() * 4, "norms");
  const size_t kv_elems = (size_t)c.max_batch * L * c.n_kv_heads * c.max_seq * hd;
  m->kv8 = (c.flags & LLM_KV_Q8) != 0;
  m->bkv8_ok = m->kv8;  // the batched attention reads and appends the int8 cache too
  if (m->kv8) {
    AL(m->d_k8, kv_elems, "int8 K cache");
    AL(m->d_v8, kv_elems, "int8 V cache");
    AL(m->d_ks, kv_elems / 32 * 2, "K cache scales");
    AL(m->d_vs, kv_elems / 32 * 2, "V cache scales");
  } else {
    AL(m->d_k, kv_elems * 2, "K cache");
    AL(m->d_v, kv_elems * 2, "V cache");
  }
  AL(m->d_rope, (size_t)c.max_seq * (hd / 2) * sizeof(float2), "rope table");

  for (int l = 0; l < L; ++l) {
    m->qkv.push_back(plan_gemv(m->mats[mi_qkv[l]], m->n_sm));
    m->wo.push_back(plan_gemv(m->mats[mi_wo[l]], m->n_sm));
    m->gu.push_back(plan_gemv(m->mats[mi_gu[l]], m->n_sm));
    m->down.push_back(plan_gemv(m->mats[mi_down[l]], m->n_sm));
  }
  m->lm = plan_gemv(m->mats[mi_lm], m->n_sm);
  // split-row-tile partials: one region per GEMV kind (QKV, WO, GU, DOWN, LM)
  // input ranges of the persistent step: 4 (else 2, else 1) equal ranges of
  // whole 64-input groups, whole heads of the attention output, and at least
  // 4 groups per range (a reduction window of the step spans at most 6 row tiles)
  m->step_R = 1;
  for (int R : {4, 2}) {
    auto ok = [&](int K) { return K % (64 * R) == 0 && K / R >= 256; };
    if (ok(d) && ok(m->q_dim) && ok(F) && (m->q_dim / R) % hd == 0 && m->n_sm >= R) {
      m->step_R = R;
      break;
    }
  }
  // Up to 4 passes over the cache, every CTA computes the attention of the kv
  // head of its o-projection range itself when that range is exactly one kv
  // head (its CTAs would otherwise run several items one after another);
  // otherwise, and for longer caches, the attention phase spreads the items.
  {
    const int hpr = c.n_kv_heads / m->step_R;
    m->step_fuse_len = (c.n_kv_heads % m->step_R == 0 && hpr == 1 && gq * hd <= kSFuseOut) ? 4 * step_attn_pp(hd) : 0;
  }
  // slots per row tile: the per-kernel path's split count or the step's ranges
  auto part_floats = [&](const GemvPlan& g) { return (size_t)g.m.n_rt * std::max(g.part.S, m->step_R) * kTileRows; };
  size_t pf[5] = {0, 0, 0, 0, part_floats(m->lm)};
  int nrt[5] = {0, 0, 0, 0, m->lm.m.n_rt};
  for (int l = 0; l < L; ++l) {
    pf[0] = std::max(pf[0], part_floats(m->qkv[l]));
    pf[1] = std::max(pf[1], part_floats(m->wo[l]));
    pf[2] = std::max(pf[2], part_floats(m->gu[l]));
    pf[3] = std::max(pf[3], part_floats(m->down[l]));
    nrt[0] = std::max(nrt[0], m->qkv[l].m.n_rt);
    nrt[1] = std::max(nrt[1], m->wo[l].m.n_rt);
    nrt[2] = std::max(nrt[2], m->gu[l].m.n_rt);
    nrt[3] = std::max(nrt[3], m->down[l].m.n_rt);
  }
  const size_t part_total = pf[0] + pf[1] + pf[2] + pf[3] + pf[4];
  const size_t cnt_total = (size_t)nrt[0] + nrt[1] + nrt[2] + nrt[3] + nrt[4] + c.n_kv_heads + 1;
  AL(m->d_part, part_total * 4, "GEMV partials");
  AL(m->d_cnt, cnt_total * 4, "counters");
  {
    float* pp = m->d_part;
    int* cc = m->d_cnt;
    std::vector<GemvPlan>* kinds[4] = {&m->qkv, &m->wo, &m->gu, &m->down};
    for (int k = 0; k < 4; ++k) {
      for (auto& g : *kinds[k]) {
        g.part_buf = pp;
        g.counters = cc;
      }
      pp += pf[k];
      cc += nrt[k];
    }
    m->lm.part_buf = pp;
    m->lm.counters = cc;
    cc += nrt[4];
    m->d_attn_cnt = cc;
    m->d_greedy_cnt = cc + c.n_kv_heads;
  }
  m->attn_P = std::max(1, m->n_sm / c.n_kv_heads);
  AL(m->d_attn_part, (size_t)c.n_kv_heads * m->attn_P * gq * (hd + 2) * 4, "attention partials");
  AL(m->d_qkv, (size_t)(m->q_dim + 2 * m->kv_dim) * 4, "q|k|v");
  AL(m->d_obuf, (size_t)m->q_dim * 4, "attention output");
  AL(m->d_abuf, (size_t)F * 4, "SwiGLU output");
  AL(m->d_xbuf, (size_t)(L + 1) * d * 4, "residual stream");
  AL(m->d_hbuf, (size_t)L * d * 4, "post-attention residual");
  AL(m->d_logits, (size_t)V * 4, "logits");
  AL(m->d_cand_v, (size_t)std::max(m->lm.part.N, m->n_sm) * 4, "greedy candidates");
  AL(m->d_cand_i, (size_t)std::max(m->lm.part.N, m->n_sm) * 4, "greedy candidates");
  // ---- the persistent step: phase table (one for every sequence)
  m->use_step = !(c.flags & LLM_MULTI_KERNEL) && step_supported(gq, hd) && d <= kSMaxDim &&
                std::min({d, m->q_dim, F}) >= 256;
  for (bool fused : {false, true}) {
    if (!m->use_step) break;
    const KernelRef k = step_kernel_ref(gq, hd, fused, (c.flags & LLM_W4A8) != 0, (c.flags & LLM_KV_Q8) != 0);
    int per_sm = 0;
    cudaError_t e = k.fn ? raise_smem_limit(k.fn, k.smem) : cudaErrorInvalidDeviceFunction;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, kSThreads, k.smem);
    if (e != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      m->use_step = false;  // fall back to the per-kernel step
    }
  }
  if (m->kv8 && !m->use_step)
    return fail(set_err(m, LLM_ERR_UNSUPPORTED,
                        "the int8 K/V cache (LLM_KV_Q8) runs in the persistent step only: not with LLM_MULTI_KERNEL, "
                        "and the shape must fit it (head_dim 64 or 128, dim, q_dim and ffn_dim >= 256)"));
  std::vector<Phase> phases;
  {
    auto gemv_phase = [&](const GemvPlan& g, float* out_part) {
      Phase ph{};
      ph.type = PH_GEMV;
      ph.units = m->d_arena + g.m.off;
      ph.n_rt = g.m.n_rt;
      ph.G = g.m.G;
      ph.K = g.m.cols;
      ph.bf16 = g.m.bf16;
      ph.unit_bytes = g.m.unit_bytes();
      ph.GR = g.m.G / m->step_R;
      ph.out_part = out_part;
      return ph;
    };
    // per-range sums of squares: 4 floats per phase (entries beyond R stay zero)
    const int n_ph = 5 * L + 2;
    AL(m->d_step_ss, (size_t)n_ph * 4 * 4, "step sums of squares");
    auto ssp = [&](int ph) { return m->d_step_ss + 4 * (size_t)ph; };
    for (int l = 0; l < L; ++l) {
      Phase q = gemv_phase(m->qkv[l], m->qkv[l].part_buf);
      q.layer = l;
      if (l == 0) {
        q.in_mode = m->embed_bf16 ? IN_EMBED_BF16 : IN_EMBED_F32;
      } else {
        q.in_mode = IN_RESID;
        q.in_part = m->down[l - 1].part_buf;
      }
      q.in_store = m->d_xbuf + (size_t)l * d;
      q.norm_w = m->d_norms + m->off_attn_norm[l];
      q.ss_out = ssp(5 * l);
      phases.push_back(q);
      Phase a{};
      a.type = PH_ATTN;
      a.layer = l;
      a.qkv_part = m->qkv[l].part_buf;
      a.ss_in = ssp(5 * l);
      a.q_norm = c.qk_norm ? m->d_norms + m->off_q_norm[l] : nullptr;
      a.k_norm = c.qk_norm ? m->d_norms + m->off_k_norm[l] : nullptr;
      phases.push_back(a);
      Phase o = gemv_phase(m->wo[l], m->wo[l].part_buf);
      o.layer = l;
      o.in_mode = IN_ATTN;
      // what the attention needs when the o-projection's build computes it
      o.qkv_part = a.qkv_part;
      o.ss_in = a.ss_in;
      o.q_norm = a.q_norm;
      o.k_norm = a.k_norm;
      phases.push_back(o);
      Phase gu = gemv_phase(m->gu[l], m->gu[l].part_buf);
      gu.layer = l;
      gu.in_mode = IN_RESID;
      gu.in_part = m->wo[l].part_buf;
      gu.in_store = m->d_hbuf + (size_t)l * d;
      gu.norm_w = m->d_norms + m->off_ffn_norm[l];
      gu.ss_out = ssp(5 * l + 3);
      phases.push_back(gu);
      Phase dn = gemv_phase(m->down[l], m->down[l].part_buf);
      dn.layer = l;
      dn.in_mode = IN_SWIGLU;
      dn.in_part = m->gu[l].part_buf;
      dn.ss_in = ssp(5 * l + 3);
      phases.push_back(dn);
    }
    Phase lmp = gemv_phase(m->lm, m->lm.part_buf);
    lmp.in_mode = IN_RESID;
    lmp.in_part = m->down[L - 1].part_buf;
    lmp.in_store = m->d_xbuf + (size_t)L * d;
    lmp.norm_w = m->d_norms + m->off_final_norm;
    lmp.ss_out = ssp(5 * L);
    phases.push_back(lmp);
    Phase lg{};
    lg.type = PH_LOGITS;
    lg.lm_part = m->lm.part_buf;
    lg.ss_in = ssp(5 * L);
    lg.vocab = V;
    phases.push_back(lg);
  }
  m->n_phases = (int)phases.size();
  AL(m->d_phases, phases.size() * sizeof(Phase), "phase table");
  AL(m->d_step_sync, 2 * sizeof(int), "step barrier");
  // ---- the dataflow step: the same GEMVs as phases whose outputs travel as
  // flagged words (one region per phase), the LM head over whole rows
  std::vector<LPhase> lph;
  {
    const int R = m->step_R;
    const int hpr = R > 0 ? c.n_kv_heads / R : 0;
    bool ok = m->use_step && (c.flags & LLM_DATAFLOW_STEP) && !(c.flags & (LLM_W4A8 | LLM_KV_Q8)) && m->n_sm <= kLMaxCTAs && R >= 1 &&
              c.n_kv_heads % R == 0 && hpr * gq * hd <= kSFuseOut && d / R <= kLMaxRes && d <= kLMaxKr;
    auto lgemv = [&](const GemvPlan& g, int r) {
      LPhase p{};
      p.units = m->d_arena + g.m.off;
      p.n_rt = g.m.n_rt;
      p.G = g.m.G;
      p.K = g.m.cols;
      p.bf16 = g.m.bf16;
      p.unit_bytes = g.m.unit_bytes();
      p.R = r;
      p.GR = g.m.G / r;
      p.NB = ll_blocks(p.n_rt, m->n_sm, r, p.GR, (kLNSlot - 1) * (kLSlotBytes / p.unit_bytes) / kLWarps);
      if (p.NB == 0 || g.m.G % r || g.m.cols / r > kLMaxKr) ok = false;
      return p;
    };
    // word counts: per layer q|k|v, o, gate|up, down partials [n_rt][R][32],
    // the two norms' range sums [4]; the last residual [dim]; the candidates [2N]
    // every region starts on a 1 KB boundary: a row tile's 32 words then fill two
    // whole cache lines, which no other CTA writes
    size_t words = 0;
    auto region = [&](size_t n) {
      const size_t o = words;
      words += (n + 127) / 128 * 128;
      return o;
    };
    std::vector<size_t> o_qkv(L), o_wo(L), o_gu(L), o_dn(L), o_ssq(L), o_ssg(L);
    for (int l = 0; l < L && ok; ++l) {
      o_qkv[l] = region((size_t)m->qkv[l].m.n_rt * R * 32);
      o_wo[l] = region((size_t)m->wo[l].m.n_rt * R * 32);
      o_gu[l] = region((size_t)m->gu[l].m.n_rt * R * 32);
      o_dn[l] = region((size_t)m->down[l].m.n_rt * R * 32);
      o_ssq[l] = region(4);
      o_ssg[l] = region(4);
    }
    const size_t o_res = region((size_t)d);
    const size_t o_cand = region(2 * (size_t)m->n_sm);
    if (ok) {
      AL(m->d_ll, words * 8, "flagged words");
      AL(m->d_epoch, 4, "step epoch");
      AL(m->d_ll_abort, 4 * (1 + (size_t)m->n_sm), "abort flag and progress");
      uint64_t* W = m->d_ll;
      for (int l = 0; l < L; ++l) {
        LPhase q = lgemv(m->qkv[l], R);
        q.layer = l;
        q.in_mode = l == 0 ? (m->embed_bf16 ? LIN_EMBED_BF16 : LIN_EMBED_F32) : LIN_RESID;
        q.in_ll = l == 0 ? nullptr : W + o_dn[l - 1];
        q.in_R = R;
        q.norm_w = m->d_norms + m->off_attn_norm[l];
        q.ss_out = W + o_ssq[l];
        q.in_store = m->d_xbuf + (size_t)l * d;
        q.out_ll = W + o_qkv[l];
        LPhase o = lgemv(m->wo[l], R);
        o.layer = l;
        o.in_mode = LIN_ATTN;
        o.in_ll = W + o_qkv[l];
        o.in_R = R;
        o.ss_in = W + o_ssq[l];
        o.q_norm = c.qk_norm ? m->d_norms + m->off_q_norm[l] : nullptr;
        o.k_norm = c.qk_norm ? m->d_norms + m->off_k_norm[l] : nullptr;
        o.out_ll = W + o_wo[l];
        LPhase gu = lgemv(m->gu[l], R);
        gu.layer = l;
        gu.in_mode = LIN_RESID;
        gu.in_ll = W + o_wo[l];
        gu.in_R = R;
        gu.norm_w = m->d_norms + m->off_ffn_norm[l];
        gu.ss_out = W + o_ssg[l];
        gu.in_store = m->d_hbuf + (size_t)l * d;
        gu.res_out = l == L - 1 ? W + o_res : nullptr;
        gu.out_ll = W + o_gu[l];
        LPhase dn = lgemv(m->down[l], R);
        dn.layer = l;
        dn.in_mode = LIN_SWIGLU;
        dn.in_ll = W + o_gu[l];
        dn.in_R = R;
        dn.ss_in = W + o_ssg[l];
        dn.out_ll = W + o_dn[l];
        lph.insert(lph.end(), {q, o, gu, dn});
      }
      LPhase lm = lgemv(m->lm, 1);
      lm.layer = -1;
      lm.in_mode = LIN_FINAL;
      lm.in_ll = W + o_dn[L - 1];
      lm.in_R = R;
      lm.res_ll = W + o_res;
      lm.norm_w = m->d_norms + m->off_final_norm;
      lm.in_store = m->d_xbuf + (size_t)L * d;
      lm.out_ll = nullptr;
      lph.push_back(lm);
      m->d_cand = W + o_cand;
    }
    if (ok) {
      const KernelRef k = stepll_kernel_ref(gq, hd);
      int per_sm = 0;
      cudaError_t e = k.fn ? raise_smem_limit(k.fn, k.smem) : cudaErrorInvalidDeviceFunction;
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, kLThreads, k.smem);
      if (e != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        ok = false;  // the barrier-synchronised step serves every call
      }
    }
    m->use_ll = ok;
    m->ll_fuse_len = ok ? 4 * step_attn_pp(hd) : 0;
    if (ok) {
      m->n_lphases = (int)lph.size();
      AL(m->d_lphases, lph.size() * sizeof(LPhase), "dataflow phase table");
      const size_t ll_bytes = words * 8;
      cudaError_t e = cudaMemset(m->d_ll, 0, ll_bytes);  // flag 0: never a step's flag
      const uint32_t one = 1;
      if (e == cudaSuccess) e = cudaMemcpy(m->d_epoch, &one, 4, cudaMemcpyHostToDevice);
      if (e == cudaSuccess) e = cudaMemset(m->d_ll_abort, 0, 4 * (1 + (size_t)m->n_sm));
      if (e == cudaSuccess)
        e = cudaMemcpy(m->d_lphases, lph.data(), lph.size() * sizeof(LPhase), cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return fail(cuda_fail(m, e, "dataflow step setup"));
      m->stamps_steps = kLStampSteps;
      AL(m->d_stamps, (size_t)kLStampSteps * m->n_lphases * m->n_sm * 16 * 8, "phase timestamps");
    }
  }
  if (LLMQ_PHASE_STAMPS && m->use_step && !m->use_ll)  // llm_phase_times on the grid-barrier step: one step
    AL(m->d_stamps, (size_t)m->n_phases * m->n_sm * 16 * 8, "phase timestamps");
  // ---- the batched pipeline (one token for every sequence of a batch, or a
  // chunk of up to kBM prompt tokens of one sequence)
  size_t bcnt_total = 0;
  {
    const int B = std::max(c.max_batch, kBM);  // rows
    size_t part_floats = 0;
    int max_blocks = 1;
    for (int l = 0; l < L; ++l) {
      m->bqkv.push_back(plan_bgemv(m->mats[mi_qkv[l]], m->n_sm));
      m->bwo.push_back(plan_bgemv(m->mats[mi_wo[l]], m->n_sm));
      m->bgu.push_back(plan_bgemv(m->mats[mi_gu[l]], m->n_sm));
      m->bdown.push_back(plan_bgemv(m->mats[mi_down[l]], m->n_sm));
    }
    m->blm = plan_bgemv(m->mats[mi_lm], m->n_sm);
    std::vector<BPlan*> all = {&m->blm};
    for (int l = 0; l < L; ++l) all.insert(all.end(), {&m->bqkv[l], &m->bwo[l], &m->bgu[l], &m->bdown[l]});
    for (BPlan* b : all) {
      if (b->ks > 1) part_floats = std::max(part_floats, (size_t)b->ks * kBM * b->m.n_rt * 32);
      max_blocks = std::max(max_blocks, b->n_blocks);
      m->bsmem_max = std::max(m->bsmem_max, b->smem);
    }
    bcnt_total = (size_t)max_blocks + (size_t)B * c.n_kv_heads + 1;
    // a bf16 LM head whose 32-token input fits in shared memory beside the
    // ring runs persistent, one CTA per SM (the candidates need one slot per CTA)
    if (m->blm.m.bf16 && m->blm.m.G % kHUC == 0) {
      int optin = 0, dev = 0;
      cudaFuncAttributes fa{};
      if (cudaGetDevice(&dev) == cudaSuccess &&
          cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
          cudaFuncGetAttributes(&fa, bhead_kernel) == cudaSuccess &&
          bhead_smem_bytes(m->blm.m.cols) + fa.sharedSizeBytes <= (size_t)optin)
        m->bhead_grid = std::min({m->n_sm, m->blm.m.n_rt, m->blm.n_blocks});
      cudaGetLastError();
    }
    AL(m->d_bx, (size_t)B * d * 4, "batched residual");
    if (c.flags & LLM_DEBUG_BATCH_HIDDEN) AL(m->d_bhid, (size_t)(L + 1) * B * d * 4, "batched hidden-state capture");
    AL(m->d_bss_x, (size_t)max_blocks * kBM * 4, "batched sums of squares");
    AL(m->d_bss_h, (size_t)max_blocks * kBM * 4, "batched sums of squares");
    AL(m->d_bh, (size_t)B * d * 4, "batched residual");
    AL(m->d_bqkv, (size_t)B * (m->q_dim + 2 * m->kv_dim) * 4, "batched q|k|v");
    AL(m->d_bx_hl, (size_t)2 * kBM * d * 2, "batched staged inputs");
    AL(m->d_bh_hl, (size_t)2 * kBM * d * 2, "batched staged inputs");
    AL(m->d_bo_hl, (size_t)2 * kBM * m->q_dim * 2, "batched staged inputs");
    AL(m->d_ba_hl, (size_t)2 * kBM * F * 2, "batched staged inputs");
    AL(m->d_blogits, (size_t)B * V * 4, "batched logits");
    AL(m->d_bpart, std::max<size_t>(part_floats, 1) * 4, "batched partials");
    AL(m->d_battn_part, (size_t)B * c.n_kv_heads * m->attn_P * gq * (hd + 2) * 4, "batched attention partials");
    AL(m->d_bcand_v, (size_t)kBM * m->blm.n_blocks * 4, "batched greedy candidates");
    AL(m->d_bcand_i, (size_t)kBM * m->blm.n_blocks * 4, "batched greedy candidates");
    AL(m->d_bcnt, bcnt_total * 4, "batched counters");
    m->d_battn_cnt = m->d_bcnt + max_blocks;
    m->d_bgreedy_cnt = m->d_battn_cnt + (size_t)B * c.n_kv_heads;
  }
  AL(m->d_pos, (size_t)c.max_batch * 4, "positions");
  AL(m->d_tok, (size_t)c.max_batch * 4, "tokens");
  AL(m->d_argmax, (size_t)c.max_batch * 4, "argmax");
  AL(m->d_hist, (size_t)c.max_seq * 4, "history");
  AL(m->d_hist_ctr, 4, "history counter");
  AL(m->d_status, 4, "status");
  AL(m->d_prompt, (size_t)c.max_seq * 4, "prompt");
  AL(m->d_samp, sizeof(SampleCfg), "sampling options");
  {
    const size_t pf = ((size_t)c.max_seq + kBM - 1) / kBM * kBM;  // prompt rows, whole chunks
    AL(m->d_pf, (3 * pf + 2 * kBM) * 4, "prompt chunk rows");
    m->pf_cap = pf;
  }
#undef AL
  {
    cudaError_t e = cudaMallocHost(&m->h_stage, kStageInts * sizeof(int));
    if (e == cudaSuccess) e = cudaMallocHost(&m->h_logits, (size_t)V * sizeof(float));
    if (e != cudaSuccess) return fail(cuda_fail(m, e, "pinned staging"));
    m->h_logits_n = V;
  }

  // ---- uploads
  auto up = [&](void* dst, const void* src, size_t bytes, const char* what) -> int {
    cudaError_t e = cudaMemcpy(dst, src, bytes, cudaMemcpyHostToDevice);
    return e == cudaSuccess ? LLM_OK : cuda_fail(m, e, what);
  };
  if ((rc = up(m->d_arena, arena.data(), arena.size(), "weight upload")) != LLM_OK) return fail(rc);
  std::vector<uint8_t>().swap(arena);
  if ((rc = up(m->d_embed, emb->data, emb_bytes, "embedding upload")) != LLM_OK) return fail(rc);
  if ((rc = up(m->d_norms, norms.data(), norms.size() * 4, "norm upload")) != LLM_OK) return fail(rc);
  if ((rc = up(m->d_phases, phases.data(), phases.size() * sizeof(Phase), "phase upload")) != LLM_OK) return fail(rc);
  {
    // cos/sin of pos * base^(-2i/hd), evaluated in double, stored as fp32
    std::vector<float2> rope((size_t)c.max_seq * (hd / 2));
    for (int pos = 0; pos < c.max_seq; ++pos)
      for (int i = 0; i < hd / 2; ++i) {
        const double ang = (double)pos * std::pow(c.rope_theta, -2.0 * i / hd);
        rope[(size_t)pos * (hd / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    if ((rc = up(m->d_rope, rope.data(), rope.size() * sizeof(float2), "rope upload")) != LLM_OK) return fail(rc);
  }
  {
    cudaError_t e = cudaMemset(m->d_cnt, 0, cnt_total * 4);
    if (e == cudaSuccess && m->d_step_ss) e = cudaMemset(m->d_step_ss, 0, (size_t)(5 * L + 2) * 16);
    if (e == cudaSuccess) e = cudaMemset(m->d_samp, 0, sizeof(SampleCfg));  // temperature 0: greedy
    for (int* z : {m->d_pos, m->d_tok, m->d_argmax})
      if (e == cudaSuccess) e = cudaMemset(z, 0, 4 * (size_t)c.max_batch);
    if (e == cudaSuccess) e = cudaMemset(m->d_hist_ctr, 0, 4);
    if (e == cudaSuccess) e = cudaMemset(m->d_status, 0, 4);
    if (e == cudaSuccess && m->d_bcnt) e = cudaMemset(m->d_bcnt, 0, bcnt_total * 4);
    if (e == cudaSuccess && m->bsmem_max)
      e = raise_smem_limit(bgemv_kernel<false>, m->bsmem_max);
    if (e == cudaSuccess && m->bsmem_max)
      e = raise_smem_limit(bgemv_kernel<true>, m->bsmem_max);
    if (e == cudaSuccess && m->bhead_grid) e = raise_smem_limit(bhead_kernel, bhead_smem_bytes(m->blm.m.cols));
    if (e == cudaSuccess) e = battn_set_smem(gq, hd);
    if (m->kv8) {
      for (int8_t* z : {m->d_k8, m->d_v8})
        if (e == cudaSuccess) e = cudaMemset(z, 0, kv_elems);
      for (uint16_t* z : {m->d_ks, m->d_vs})
        if (e == cudaSuccess) e = cudaMemset(z, 0, kv_elems / 32 * 2);
    } else {
      if (e == cudaSuccess) e = cudaMemset(m->d_k, 0, kv_elems * 2);
      if (e == cudaSuccess) e = cudaMemset(m->d_v, 0, kv_elems * 2);
    }
    size_t smax = m->lm.smem;
    for (int l = 0; l < L; ++l)
      smax = std::max({smax, m->qkv[l].smem, m->wo[l].smem, m->gu[l].smem, m->down[l].smem});
    if (e == cudaSuccess)
      e = raise_smem_limit(gemv_kernel<false>, smax);
    if (e == cudaSuccess)
      e = raise_smem_limit(gemv_kernel<true>, smax);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(cuda_fail(m, e, "initialisation"));
  }
  m->len.assign(c.max_batch, 0);
  m->graphs.assign(2 * (size_t)c.max_batch, nullptr);  // per sequence: split, fused variant
  m->kernels_per_step = (m->use_step || m->use_ll) ? 1 : 5 * L + 1;
  *out = m;
  return LLM_OK;
}

int llm_decode_step(llm_model* m, int32_t seq, int32_t token, float* logits_out, int32_t* argmax_out) {
  NvtxRange nvtx_("llm_decode_step");
  int rc = check_model(m, seq);
  if (rc) return rc;
  if (token < 0 || token >= m->cfg.vocab) return set_err(m, LLM_ERR_INVALID_ARG, "token out of range");
  if (m->len[seq] + 1 > m->cfg.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "sequence is at max_seq");
  // an asynchronous call uploads from its pageable argument (staged at call
  // time, so back-to-back calls cannot race); a synchronous one via pinned memory
  const bool sync_call = host_outputs(logits_out, argmax_out);
  const int32_t tok_host = token;
  if ((rc = upload_tokens(m, m->d_tok + seq, &tok_host, 1, sync_call, kStageTok)) != LLM_OK) return rc;
  if (ll_covers(m, m->len[seq], 1)) {
    CK(enqueue_ll(m, seq, 1, 0, nullptr), "step launch");
  } else if ((rc = run_step(m, seq, m->len[seq])) != LLM_OK) {
    return rc;
  }
  m->len[seq] += 1;
  return finish_call(m, logits_out, m->d_logits, (size_t)m->cfg.vocab, argmax_out, m->d_argmax + seq, 1);
}

int llm_prefill(llm_model* m, int32_t seq, const int32_t* tokens, int32_t n, float* logits_out, int32_t* argmax_out) {
  NvtxRange nvtx_("llm_prefill");
  int rc = check_model(m, seq);
  if (rc) return rc;
  if (!tokens || n <= 0) return set_err(m, LLM_ERR_INVALID_ARG, "empty prompt");
  if (m->len[seq] + n > m->cfg.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "prompt would exceed max_seq");
  std::vector<int32_t> host_toks(n);
  CK(cudaMemcpy(host_toks.data(), tokens, (size_t)n * 4, cudaMemcpyDefault), "prompt read");
  for (int i = 0; i < n; ++i)
    if (host_toks[i] < 0 || host_toks[i] >= m->cfg.vocab)
      return set_err(m, LLM_ERR_INVALID_ARG, "prompt token out of range");
  CK(cudaMemcpyAsync(m->d_prompt, host_toks.data(), (size_t)n * 4, cudaMemcpyHostToDevice, m->stream), "prompt upload");
  if (ll_covers(m, m->len[seq], n)) {
    CK(enqueue_ll(m, seq, n, n, m->d_prompt), "prefill launch");  // every step's token forced
  } else {
    for (int i = 0; i < n; ++i) {
      CK(cudaMemcpyAsync(m->d_tok + seq, m->d_prompt + i, 4, cudaMemcpyDeviceToDevice, m->stream), "token copy");
      if ((rc = run_step(m, seq, m->len[seq] + i)) != LLM_OK) return rc;
    }
  }
  m->len[seq] += n;
  if ((rc = finish_call(m, logits_out, m->d_logits, (size_t)m->cfg.vocab, argmax_out, m->d_argmax + seq, 1)) !=
      LLM_OK)
    return rc;
  CK(cudaStreamSynchronize(m->stream), "prefill sync");  // host_toks outlives the upload
  return check_status(m);
}

int llm_prefill_batched(llm_model* m, int32_t seq, const int32_t* tokens, int32_t n, float* logits_out,
                        int32_t* argmax_out) {
  NvtxRange nvtx_("llm_prefill_batched");
  int rc = check_model(m, seq);
  if (rc) return rc;
  if (m->kv8 && !m->bkv8_ok) return set_err(m, LLM_ERR_UNSUPPORTED, "batched prompt processing with the int8 K/V cache");
  if (!tokens || n <= 0) return set_err(m, LLM_ERR_INVALID_ARG, "empty prompt");
  if (m->len[seq] + n > m->cfg.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "prompt would exceed max_seq");
  std::vector<int32_t> rows(3 * m->pf_cap);  // [tok | pos | seq]
  CK(cudaMemcpy(rows.data(), tokens, (size_t)n * 4, cudaMemcpyDefault), "prompt read");
  for (int i = 0; i < n; ++i) {
    if (rows[i] < 0 || rows[i] >= m->cfg.vocab) return set_err(m, LLM_ERR_INVALID_ARG, "prompt token out of range");
    rows[m->pf_cap + i] = m->len[seq] + i;
    rows[2 * m->pf_cap + i] = seq;
  }
  CK(cudaMemcpyAsync(m->d_pf, rows.data(), rows.size() * 4, cudaMemcpyHostToDevice, m->stream), "prompt rows upload");
  int* scratch = m->d_pf + 3 * m->pf_cap;  // [kBM] greedy tokens, [kBM] argmax of the last chunk
  int last_rows = 0;
  for (int c0 = 0; c0 < n; c0 += kBM) {
    BatchedIO io{};
    io.M = std::min(kBM, n - c0);
    io.tok = m->d_pf + c0;
    io.pos = m->d_pf + m->pf_cap + c0;
    io.seq = m->d_pf + 2 * m->pf_cap + c0;
    io.chunk = true;
    io.lm = c0 + io.M == n;  // logits of the prompt's last token only
    io.tok_io = scratch;
    io.argmax_out = scratch + kBM;
    last_rows = io.M;
    CK(enqueue_batched(m, io), "prompt chunk launch");
  }
  if (m->sampling)  // the last row's logits; its position counter was advanced by the greedy epilogue
    CK(launch_sample(m, seq, m->d_blogits + (size_t)(last_rows - 1) * m->cfg.vocab, m->d_pf + m->pf_cap + n - 1,
                     nullptr, scratch + kBM + last_rows - 1, false),
       "sampling launch");
  m->len[seq] += n;
  const int32_t next_pos = m->len[seq];  // the decode steps' position counter (pageable: staged at call time)
  CK(cudaMemcpyAsync(m->d_pos + seq, &next_pos, 4, cudaMemcpyHostToDevice, m->stream), "position update");
  bool host = false;
  if ((rc = copy_out(m, logits_out, m->d_blogits + (size_t)(last_rows - 1) * m->cfg.vocab,
                     (size_t)m->cfg.vocab * 4, &host)) != LLM_OK)
    return rc;
  if ((rc = copy_out(m, argmax_out, scratch + kBM + last_rows - 1, 4, &host)) != LLM_OK) return rc;
  CK(cudaStreamSynchronize(m->stream), "prefill sync");  // `rows` outlives the upload
  return check_status(m);
}

int llm_set_sampling(llm_model* m, float temperature, int32_t top_k, float top_p, uint64_t seed) {
  int rc = check_model(m, 0);
  if (rc) return rc;
  if (!(temperature >= 0.f) || !(temperature < INFINITY))
    return set_err(m, LLM_ERR_INVALID_ARG, "temperature must be finite and >= 0");
  if (temperature > 0.f && (top_k < 1 || top_k > kSampleMaxK))
    return set_err(m, LLM_ERR_INVALID_ARG, "top_k must be in 1..64 when sampling");
  if (temperature > 0.f && !(top_p > 0.f && top_p <= 1.f))
    return set_err(m, LLM_ERR_INVALID_ARG, "top_p must be in (0, 1]");
  SampleCfg h{};
  h.temperature = temperature;
  h.top_p = top_p;
  h.top_k = top_k;
  h.seed_lo = (uint32_t)(seed & 0xFFFFFFFFull);
  h.seed_hi = (uint32_t)(seed >> 32);
  CK(cudaStreamSynchronize(m->stream), "sampling sync");  // no step in flight reads the options
  CK(cudaMemcpy(m->d_samp, &h, sizeof(h), cudaMemcpyHostToDevice), "sampling upload");
  const bool on = temperature > 0.f;
  if (on != m->sampling) {  // the captured steps gain or lose the sampling kernel: capture again
    for (auto& g : m->graphs)
      if (g) {
        cudaGraphExecDestroy(g);
        g = nullptr;
      }
    m->sampling = on;
  }
  return LLM_OK;
}

int llm_decode_greedy(llm_model* m, int32_t seq, int32_t first_token, int32_t n_steps, int32_t* tokens_out) {
  NvtxRange nvtx_("llm_decode_greedy");
  int rc = check_model(m, seq);
  if (rc) return rc;
  if (n_steps <= 0 || !tokens_out) return set_err(m, LLM_ERR_INVALID_ARG, "n_steps <= 0 or null tokens_out");
  if (first_token < 0 || first_token >= m->cfg.vocab) return set_err(m, LLM_ERR_INVALID_ARG, "token out of range");
  if (m->len[seq] + n_steps > m->cfg.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "steps would exceed max_seq");
  const int32_t tok_host = first_token;
  if ((rc = upload_tokens(m, m->d_tok + seq, &tok_host, 1, host_outputs(tokens_out, nullptr), kStageTok)) != LLM_OK)
    return rc;
  CK(cudaMemsetAsync(m->d_hist_ctr, 0, 4, m->stream), "history reset");
  // the steps the dataflow kernel covers go in one launch, the rest step by step
  int done = 0;
  if (m->use_ll && !m->sampling) {
    const int n1 = std::min(n_steps, m->ll_fuse_len - m->len[seq]);
    if (n1 > 0) {
      CK(enqueue_ll(m, seq, n1, 0, nullptr), "greedy launch");
      done = n1;
    }
  }
  for (int i = done; i < n_steps; ++i)
    if ((rc = run_step(m, seq, m->len[seq] + i)) != LLM_OK) return rc;
  m->len[seq] += n_steps;
  return finish_call(m, nullptr, nullptr, 0, tokens_out, m->d_hist, (size_t)n_steps);
}

int llm_decode_step_batch(llm_model* m, const int32_t* tokens, int32_t n_seq, float* logits_out, int32_t* argmax_out) {
  NvtxRange nvtx_("llm_decode_step_batch");
  int rc = check_model(m, 0);
  if (rc) return rc;
  if (m->kv8 && !m->bkv8_ok) return set_err(m, LLM_ERR_UNSUPPORTED, "batched decode with the int8 K/V cache");
  const llm_config& c = m->cfg;
  if (c.max_batch < 2) return set_err(m, LLM_ERR_UNSUPPORTED, "the model was created with max_batch < 2");
  if (n_seq != c.max_batch) return set_err(m, LLM_ERR_INVALID_ARG, "n_seq must equal max_batch");
  for (int b = 0; b < n_seq; ++b)
    if (m->len[b] + 1 > c.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "a sequence is at max_seq");
  std::vector<int32_t> host_toks;
  if (tokens) {  // else: each sequence continues from its previous greedy token, on the device
    host_toks.resize(n_seq);
    CK(cudaMemcpy(host_toks.data(), tokens, (size_t)n_seq * 4, cudaMemcpyDefault), "token read");
    for (int b = 0; b < n_seq; ++b)
      if (host_toks[b] < 0 || host_toks[b] >= c.vocab) return set_err(m, LLM_ERR_INVALID_ARG, "token out of range");
    // a call given tokens synchronizes before it returns: the pinned slot is free again by then
    if ((rc = upload_tokens(m, m->d_tok, host_toks.data(), n_seq, true, kStageToks)) != LLM_OK) return rc;
  }
  if (c.flags & LLM_NO_GRAPH) {
    CK(enqueue_batched(m, decode_io(m)), "batched step launch");
  } else {
    if (!m->bgraph) {
      cudaGraph_t g = nullptr;
      CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal), "begin capture");
      cudaError_t e = enqueue_batched(m, decode_io(m));
      cudaError_t e2 = cudaStreamEndCapture(m->stream, &g);
      if (e != cudaSuccess) return cuda_fail(m, e, "batched step capture");
      if (e2 != cudaSuccess) return cuda_fail(m, e2, "end capture");
      e = cudaGraphInstantiate(&m->bgraph, g, 0);
      cudaGraphDestroy(g);
      if (e != cudaSuccess) return cuda_fail(m, e, "graph instantiate");
    }
    CK(cudaGraphLaunch(m->bgraph, m->stream), "graph launch");
  }
  for (int b = 0; b < n_seq; ++b) m->len[b] += 1;
  const bool host = host_outputs(logits_out, argmax_out);
  if ((rc = finish_call(m, logits_out, m->d_blogits, (size_t)n_seq * c.vocab, argmax_out, m->d_argmax,
                        (size_t)n_seq)) != LLM_OK)
    return rc;
  if (tokens && !host) return check_status(m);
  return LLM_OK;
}

int llm_kv_reset(llm_model* m, int32_t seq) {
  if (!m) return set_err(nullptr, LLM_ERR_INVALID_ARG, "model is NULL");
  if (m->poisoned) return m->poisoned;
  if (seq < -1 || seq >= m->cfg.max_batch) return set_err(m, LLM_ERR_INVALID_ARG, "seq out of range");
  for (int s = 0; s < m->cfg.max_batch; ++s)
    if (seq == -1 || s == seq) {
      m->len[s] = 0;
      CK(cudaMemsetAsync(m->d_pos + s, 0, 4, m->stream), "position reset");
    }
  return LLM_OK;
}

// The cache's grouped int8 quantizer on the host (llm_kv_write into an int8
// cache): each 32 values of a (position, head) row get the fp16 scale
// fp16(amax / 127) and codes round(x / scale), half away from zero, clamped
// to +-127 -- in fp32, the operations of the kernels' append.
static void q8_quantize_host(const uint16_t* bf16, size_t n_vals, int8_t* codes, uint16_t* scales) {
  for (size_t g = 0; g < n_vals / 32; ++g) {
    float x[32], amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
      const uint32_t u = (uint32_t)bf16[g * 32 + i] << 16;
      std::memcpy(&x[i], &u, 4);
      amax = std::max(amax, std::fabs(x[i]));
    }
    const __half dh = __float2half_rn(amax / 127.0f);
    const float d = __half2float(dh);
    for (int i = 0; i < 32; ++i) {
      const float cf = d == 0.0f ? 0.0f : std::min(std::max(std::roundf(x[i] / d), -127.0f), 127.0f);
      codes[g * 32 + i] = (int8_t)(int)cf;
    }
    std::memcpy(&scales[g], &dh, 2);
  }
}

static int kv_copy(llm_model* m, int32_t seq, int32_t layer, int32_t pos0, int32_t n, const uint16_t* src_k,
                   const uint16_t* src_v, uint16_t* dst_k, uint16_t* dst_v, bool write) {
  int rc = check_model(m, seq);
  if (rc) return rc;
  const llm_config& c = m->cfg;
  if (layer < 0 || layer >= c.n_layers || pos0 < 0 || n <= 0) return set_err(m, LLM_ERR_INVALID_ARG, "bad layer/pos/n");
  if (pos0 + n > c.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "positions beyond max_seq");
  const int hd = c.head_dim, H = c.n_kv_heads;
  const size_t base = (((size_t)seq * c.n_layers + layer) * H) * c.max_seq * hd;
  if (m->kv8) {
    if (!write) return set_err(m, LLM_ERR_UNSUPPORTED, "the int8 K/V cache is read with llm_kv_read_q8");
    if (!src_k || !src_v) return set_err(m, LLM_ERR_INVALID_ARG, "null key/value pointer");
    const size_t nv = (size_t)n * H * hd;
    std::vector<uint16_t> hb(nv);
    std::vector<int8_t> codes(nv);
    std::vector<uint16_t> scales(nv / 32);
    for (int which = 0; which < 2; ++which) {
      CK(cudaMemcpy(hb.data(), which ? src_v : src_k, nv * 2, cudaMemcpyDefault), "kv read-in");
      q8_quantize_host(hb.data(), nv, codes.data(), scales.data());
      for (int g = 0; g < H; ++g) {
        const size_t off = base + ((size_t)g * c.max_seq + pos0) * hd;
        CK(cudaMemcpy2D((which ? m->d_v8 : m->d_k8) + off, hd, codes.data() + (size_t)g * hd, (size_t)H * hd, hd, n,
                        cudaMemcpyHostToDevice), "kv write");
        CK(cudaMemcpy2D((which ? m->d_vs : m->d_ks) + off / 32, hd / 16, scales.data() + (size_t)g * (hd / 32),
                        (size_t)H * (hd / 16), hd / 16, n, cudaMemcpyHostToDevice), "kv scale write");
      }
    }
    m->len[seq] = std::max(m->len[seq], pos0 + n);
    m->h_stage[1] = m->len[seq];
    CK(cudaMemcpyAsync(m->d_pos + seq, m->h_stage + 1, 4, cudaMemcpyHostToDevice, m->stream), "position set");
    CK(cudaStreamSynchronize(m->stream), "kv sync");
    return LLM_OK;
  }
  for (int g = 0; g < H; ++g) {
    const size_t cache_off = base + ((size_t)g * c.max_seq + pos0) * hd;
    for (int which = 0; which < 2; ++which) {
      uint16_t* cache = (which ? m->d_v : m->d_k) + cache_off;
      if (write) {
        const uint16_t* s = (which ? src_v : src_k);
        if (!s) return set_err(m, LLM_ERR_INVALID_ARG, "null key/value pointer");
        CK(cudaMemcpy2DAsync(cache, hd * 2, s + (size_t)g * hd, (size_t)H * hd * 2, hd * 2, n, cudaMemcpyDefault,
                             m->stream), "kv write");
      } else {
        uint16_t* dd = (which ? dst_v : dst_k);
        if (!dd) return set_err(m, LLM_ERR_INVALID_ARG, "null key/value pointer");
        CK(cudaMemcpy2DAsync(dd + (size_t)g * hd, (size_t)H * hd * 2, cache, hd * 2, hd * 2, n, cudaMemcpyDefault,
                             m->stream), "kv read");
      }
    }
  }
  if (write) {
    m->len[seq] = std::max(m->len[seq], pos0 + n);
    m->h_stage[1] = m->len[seq];
    CK(cudaMemcpyAsync(m->d_pos + seq, m->h_stage + 1, 4, cudaMemcpyHostToDevice, m->stream), "position set");
  }
  CK(cudaStreamSynchronize(m->stream), "kv sync");
  return LLM_OK;
}

int llm_kv_write(llm_model* m, int32_t seq, int32_t layer, int32_t pos0, int32_t n, const uint16_t* k,
                 const uint16_t* v) {
  return kv_copy(m, seq, layer, pos0, n, k, v, nullptr, nullptr, true);
}

int llm_kv_read(llm_model* m, int32_t seq, int32_t layer, int32_t pos0, int32_t n, uint16_t* k, uint16_t* v) {
  return kv_copy(m, seq, layer, pos0, n, nullptr, nullptr, k, v, false);
}

int llm_kv_read_q8(llm_model* m, int32_t seq, int32_t layer, int32_t pos0, int32_t n, int8_t* k, uint16_t* ks,
                   int8_t* v, uint16_t* vs) {
  int rc = check_model(m, seq);
  if (rc) return rc;
  const llm_config& c = m->cfg;
  if (!m->kv8) return set_err(m, LLM_ERR_UNSUPPORTED, "the model's K/V cache is bf16 (llm_kv_read)");
  if (!k || !ks || !v || !vs) return set_err(m, LLM_ERR_INVALID_ARG, "null output");
  if (layer < 0 || layer >= c.n_layers || pos0 < 0 || n <= 0) return set_err(m, LLM_ERR_INVALID_ARG, "bad layer/pos/n");
  if (pos0 + n > c.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "positions beyond max_seq");
  const int hd = c.head_dim, H = c.n_kv_heads;
  const size_t base = (((size_t)seq * c.n_layers + layer) * H) * c.max_seq * hd;
  for (int g = 0; g < H; ++g) {
    const size_t off = base + ((size_t)g * c.max_seq + pos0) * hd;
    for (int which = 0; which < 2; ++which) {
      CK(cudaMemcpy2DAsync((which ? v : k) + (size_t)g * hd, (size_t)H * hd, (which ? m->d_v8 : m->d_k8) + off, hd, hd,
                           n, cudaMemcpyDefault, m->stream), "kv read");
      CK(cudaMemcpy2DAsync((which ? vs : ks) + (size_t)g * (hd / 32), (size_t)H * (hd / 16),
                           (which ? m->d_vs : m->d_ks) + off / 32, hd / 16, hd / 16, n, cudaMemcpyDefault, m->stream),
         "kv scale read");
    }
  }
  CK(cudaStreamSynchronize(m->stream), "kv sync");
  return LLM_OK;
}

int llm_kv_len(const llm_model* m, int32_t seq) {
  if (!m) return LLM_ERR_INVALID_ARG;
  if (seq < 0 || seq >= m->cfg.max_batch) return LLM_ERR_INVALID_ARG;
  return m->len[seq];
}

int llm_debug_hidden(llm_model* m, float* out) {
  int rc = check_model(m, 0);
  if (rc) return rc;
  if (!out) return set_err(m, LLM_ERR_INVALID_ARG, "null output");
  CK(cudaMemcpyAsync(out, m->d_xbuf, (size_t)(m->cfg.n_layers + 1) * m->cfg.dim * 4, cudaMemcpyDefault, m->stream),
     "hidden copy");
  CK(cudaStreamSynchronize(m->stream), "hidden sync");
  return LLM_OK;
}

int llm_debug_hidden_batch(llm_model* m, float* out) {
  int rc = check_model(m, 0);
  if (rc) return rc;
  if (!out) return set_err(m, LLM_ERR_INVALID_ARG, "null output");
  if (!m->d_bhid) return set_err(m, LLM_ERR_UNSUPPORTED, "the model was not created with LLM_DEBUG_BATCH_HIDDEN");
  const size_t n = (size_t)(m->cfg.n_layers + 1) * m->cfg.max_batch * m->cfg.dim;
  CK(cudaMemcpyAsync(out, m->d_bhid, n * 4, cudaMemcpyDefault, m->stream), "hidden copy");
  CK(cudaStreamSynchronize(m->stream), "hidden sync");
  return LLM_OK;
}

int llm_debug_fail_alloc(int32_t nth) {
  g_fail_alloc.store(nth > 0 ? nth : 0);
  return LLM_OK;
}

int llm_debug_unpack(llm_model* m, const char* name, uint8_t* codes, uint16_t* scales, uint16_t* mins) {
  int rc = check_model(m, 0);
  if (rc) return rc;
  if (!name || !codes || !scales || !mins) return set_err(m, LLM_ERR_INVALID_ARG, "null argument");
  auto it = m->places.find(name);
  if (it == m->places.end()) return set_err(m, LLM_ERR_NOT_FOUND, std::string("no 4-bit tensor named ") + name);
  const Mat& x = m->mats[it->second.mat];
  const auto shp = m->shapes[name];
  std::vector<uint8_t> units(x.bytes());
  CK(cudaMemcpy(units.data(), m->d_arena + x.off, x.bytes(), cudaMemcpyDeviceToHost), "unpack copy");
  std::memset(codes, 0, (size_t)shp.first * shp.second / 2);
  unpack_q4(units.data(), x.G, codes, scales, mins, (int)shp.first, (int)shp.second, it->second.kind, it->second.row0);
  return LLM_OK;
}

int llm_model_stats(const llm_model* m, llm_stats* out) {
  if (!m || !out) return LLM_ERR_INVALID_ARG;
  out->device_bytes = (int64_t)m->device_bytes;
  int64_t w = 0;
  for (const auto& x : m->mats) w += (int64_t)x.bytes();
  out->weight_stream_bytes = w;
  out->kv_bytes_per_pos = m->kv8 ? (int64_t)2 * m->cfg.n_layers * m->cfg.n_kv_heads * (m->cfg.head_dim + m->cfg.head_dim / 16)
                                 : (int64_t)2 * m->cfg.n_layers * m->cfg.n_kv_heads * m->cfg.head_dim * 2;
  out->kernels_per_step = m->kernels_per_step;
  out->n_sm = m->n_sm;
  return LLM_OK;
}

int llm_profile_step(llm_model* m, int32_t seq, int32_t token, llm_kernel_time* out, int32_t max_out) {
  int rc = check_model(m, seq);
  if (rc) return rc;
  if (m->kv8) return set_err(m, LLM_ERR_UNSUPPORTED, "the per-kernel profile runs the bf16 K/V cache's kernels");
  if (token < 0 || token >= m->cfg.vocab) return set_err(m, LLM_ERR_INVALID_ARG, "token out of range");
  if (m->len[seq] + 1 > m->cfg.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "sequence is at max_seq");
  if (!out || max_out < 0) return set_err(m, LLM_ERR_INVALID_ARG, "null output");
  const int32_t tok_host = token;
  CK(cudaMemcpyAsync(m->d_tok + seq, &tok_host, 4, cudaMemcpyHostToDevice, m->stream), "token upload");
  Prof prof;
  prof.kv_len = m->len[seq] + 1;
  cudaError_t e = enqueue_step(m, seq, &prof);
  if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
  for (size_t i = 0; e == cudaSuccess && i < prof.rec.size(); ++i)
    e = cudaEventElapsedTime(&prof.rec[i].ms, prof.ev[2 * i], prof.ev[2 * i + 1]);
  for (auto ev : prof.ev) cudaEventDestroy(ev);
  if (e != cudaSuccess) return cuda_fail(m, e, "profile step");
  m->len[seq] += 1;
  const int n = (int)prof.rec.size();
  for (int i = 0; i < n && i < max_out; ++i) out[i] = prof.rec[i];
  rc = check_status(m);
  return rc ? rc : n;
}

int llm_time_kernel(llm_model* m, int32_t seq, int32_t which, int32_t layer, int32_t n, float* ms,
                    int64_t* bytes) {
  int rc = check_model(m, seq);
  if (rc) return rc;
  const int L = m->cfg.n_layers;
  if (which < 0 || which > 6 || n <= 0 || !ms || !bytes) return set_err(m, LLM_ERR_INVALID_ARG, "bad kernel/n");
  if (layer < -1 || layer >= L) return set_err(m, LLM_ERR_INVALID_ARG, "bad layer");
  if (m->len[seq] < 1) return set_err(m, LLM_ERR_INVALID_ARG, "run a step of the sequence first");
  if (m->kv8 && which == W_ATTN)
    return set_err(m, LLM_ERR_UNSUPPORTED, "the per-kernel attention reads the bf16 K/V cache");
  // attention re-reads position len-1 (and re-appends that slot with the values already there)
  m->h_stage[2] = m->len[seq] - 1;
  CK(cudaMemcpyAsync(m->d_pos + seq, m->h_stage + 2, 4, cudaMemcpyHostToDevice, m->stream), "position set");
  // launch list: one kernel kind over the layers (or one layer), or every 4-bit GEMV of a step
  std::vector<std::pair<int, int>> seqn;
  if (which == 6) {
    for (int l = 0; l < L; ++l)
      for (int w : {W_QKV, W_WO, W_GU, W_DOWN}) seqn.push_back({w, l});
    seqn.push_back({W_LM, 0});
  } else if (which == W_LM) {
    seqn.push_back({W_LM, 0});
  } else {
    for (int l = (layer < 0 ? 0 : layer); l < (layer < 0 ? L : layer + 1); ++l) seqn.push_back({which, l});
  }
  int64_t total_bytes = 0;
  for (auto& x : seqn) total_bytes += launch_bytes(m, x.first, x.second, m->len[seq]);
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0), "event");
  CK(cudaEventCreate(&e1), "event");
  cudaError_t e = launch_one(m, seq, seqn[0].first, seqn[0].second, false);  // warm, no programmatic edge
  if (e == cudaSuccess) e = cudaEventRecord(e0, m->stream);
  for (int i = 0; e == cudaSuccess && i < n; ++i)
    for (size_t j = 0; e == cudaSuccess && j < seqn.size(); ++j)
      e = launch_one(m, seq, seqn[j].first, seqn[j].second, !(m->cfg.flags & LLM_NO_PDL));
  if (e == cudaSuccess) e = cudaEventRecord(e1, m->stream);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float t = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return cuda_fail(m, e, "kernel timing");
  m->h_stage[2] = m->len[seq];
  CK(cudaMemcpyAsync(m->d_pos + seq, m->h_stage + 2, 4, cudaMemcpyHostToDevice, m->stream), "position restore");
  *ms = t / (float)(n * seqn.size());
  *bytes = total_bytes / (int64_t)seqn.size();
  return check_status(m);
}

int llm_phase_times(llm_model* m, int32_t seq, int32_t first_token, int32_t n_steps, uint64_t* out,
                    int64_t max_out) {
  int rc = check_model(m, seq);
  if (rc) return rc;
  if (!m->use_ll) {
    // the grid-barrier step: one step per launch, [phase][CTA][16]
    if (!m->use_step) return set_err(m, LLM_ERR_UNSUPPORTED, "no persistent step on this model");
    if (!m->d_stamps)
      return set_err(m, LLM_ERR_UNSUPPORTED, "the grid-barrier step records stamps in a build with LLMQ_PHASE_STAMPS=1");
    if (n_steps != 1 || !out) return set_err(m, LLM_ERR_INVALID_ARG, "one step at a time on the grid-barrier step");
    if (first_token < 0 || first_token >= m->cfg.vocab) return set_err(m, LLM_ERR_INVALID_ARG, "token out of range");
    if (m->len[seq] + 1 > m->cfg.max_seq) return set_err(m, LLM_ERR_CTX_FULL, "sequence at max_seq");
    if (m->sampling) return set_err(m, LLM_ERR_UNSUPPORTED, "sampling on");
    const int64_t n = (int64_t)m->n_phases * m->n_sm * 16;
    if (max_out < n) return set_err(m, LLM_ERR_INVALID_ARG, "output too small");
    const bool fused = m->len[seq] + 1 <= m->step_fuse_len;
    const int32_t tok_host = first_token;
    CK(cudaMemcpyAsync(m->d_tok + seq, &tok_host, 4, cudaMemcpyHostToDevice, m->stream), "token upload");
    CK(cudaMemsetAsync(m->d_stamps, 0, (size_t)n * 8, m->stream), "timestamp reset");
    CK(enqueue_persistent_step(m, seq, fused, m->d_stamps), "profiled launch");
    m->len[seq] += 1;
    CK(cudaMemcpyAsync(out, m->d_stamps, (size_t)n * 8, cudaMemcpyDeviceToHost, m->stream), "timestamps");
    CK(cudaStreamSynchronize(m->stream), "profile sync");
    rc = check_status(m);
    return rc ? rc : (int)(n / 16);
  }
  if (n_steps <= 0 || n_steps > (int)m->stamps_steps || !out)
    return set_err(m, LLM_ERR_INVALID_ARG, "n_steps outside 1..8 or null output");
  if (first_token < 0 || first_token >= m->cfg.vocab) return set_err(m, LLM_ERR_INVALID_ARG, "token out of range");
  if (!ll_covers(m, m->len[seq], n_steps))
    return set_err(m, LLM_ERR_UNSUPPORTED, "positions beyond the flag-synchronised step's range (or sampling on)");
  const int64_t n = (int64_t)n_steps * m->n_lphases * m->n_sm * 16;
  if (max_out < n) return set_err(m, LLM_ERR_INVALID_ARG, "output too small");
  const int32_t tok_host = first_token;
  CK(cudaMemcpyAsync(m->d_tok + seq, &tok_host, 4, cudaMemcpyHostToDevice, m->stream), "token upload");
  CK(cudaMemsetAsync(m->d_stamps, 0, (size_t)n * 8, m->stream), "timestamp reset");
  CK(enqueue_ll(m, seq, n_steps, 0, nullptr, m->d_stamps), "profiled launch");
  m->len[seq] += n_steps;
  CK(cudaMemcpyAsync(out, m->d_stamps, (size_t)n * 8, cudaMemcpyDeviceToHost, m->stream), "timestamps");
  CK(cudaStreamSynchronize(m->stream), "profile sync");
  rc = check_status(m);
  return rc ? rc : (int)(n / 16);
}

int llm_sync(llm_model* m) {
  if (!m) return set_err(nullptr, LLM_ERR_INVALID_ARG, "model is NULL");
  return check_status(m);
}

static int op_matvec(const llm_tensor* w, const float* x, float* y, bool w4a8) {
  if (!w || !x || !y) return set_err(nullptr, LLM_ERR_INVALID_ARG, "null argument");
  const bool bf16 = w->dtype == LLM_BF16;
  if (w4a8 && bf16) return set_err(nullptr, LLM_ERR_UNSUPPORTED, "W4A8 needs a Q4G64 tensor");
  if (!bf16 && w->dtype != LLM_Q4G64) return set_err(nullptr, LLM_ERR_UNSUPPORTED, "dtype must be Q4G64 or BF16");
  if (w->rows <= 0 || w->cols <= 0 || w->cols % 64 || w->cols > kMaxK || w->rows > (1 << 24))
    return set_err(nullptr, LLM_ERR_UNSUPPORTED, "rows > 0 and cols a multiple of 64 up to 8192 required");
  int n_sm = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "no CUDA device");
  Mat mat;
  mat.rows = (int)w->rows;
  mat.cols = (int)w->cols;
  mat.n_rt = (mat.rows + 31) / 32;
  mat.G = mat.cols / (bf16 ? kBF16UnitCols : 64);
  mat.bf16 = bf16;
  std::vector<uint8_t> units(mat.bytes(), 0);
  if (bf16)
    repack_bf16(units.data(), mat.G, static_cast<const uint16_t*>(w->data), mat.rows, mat.cols);
  else
    repack_q4(units.data(), mat.G, static_cast<const uint8_t*>(w->codes), static_cast<const uint16_t*>(w->scales),
              static_cast<const uint16_t*>(w->mins), mat.rows, mat.cols, 0, 0);
  GemvPlan g = plan_gemv(mat, n_sm);
  uint8_t* d_units = nullptr;
  float *d_x = nullptr, *d_y = nullptr, *d_part = nullptr;
  int *d_status = nullptr, *d_cnt = nullptr;
  const size_t part_bytes = (size_t)mat.n_rt * g.part.S * kTileRows * 4;
  e = cudaMalloc(&d_units, units.size());
  if (e == cudaSuccess) e = cudaMalloc(&d_x, (size_t)mat.cols * 4);
  if (e == cudaSuccess) e = cudaMalloc(&d_y, (size_t)mat.rows * 4);
  if (e == cudaSuccess) e = cudaMalloc(&d_part, part_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&d_cnt, (size_t)mat.n_rt * 4);
  if (e == cudaSuccess) e = cudaMalloc(&d_status, 4);
  if (e == cudaSuccess) e = cudaMemcpy(d_units, units.data(), units.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(d_x, x, (size_t)mat.cols * 4, cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemset(d_status, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(d_cnt, 0, (size_t)mat.n_rt * 4);
  if (e == cudaSuccess)
    e = bf16 ? raise_smem_limit(gemv_kernel<true>, g.smem) : raise_smem_limit(gemv_kernel<false>, g.smem);
  int st = 0;
  if (e == cudaSuccess) {
    GemvParams p{};
    p.units = d_units;
    p.n_rt = mat.n_rt;
    p.G = mat.G;
    p.K = mat.cols;
    p.rows = mat.rows;
    p.unit_bytes = mat.unit_bytes();
    p.nslot = g.nslot;
    p.ring_bytes = g.ring;
    p.part = g.part;
    p.vec_mode = VEC_PLAIN;
    p.vin = d_x;
    p.w4a8 = w4a8 ? 1 : 0;
    p.epi = EPI_STORE;
    p.out = d_y;
    p.part_buf = d_part;
    p.counters = d_cnt;
    p.status = d_status;
    e = launch(bf16 ? gemv_kernel<true> : gemv_kernel<false>, dim3(g.part.N), dim3(kGemvThreads), g.smem, 0, false, p);
    if (e == cudaSuccess) e = cudaMemcpy(y, d_y, (size_t)mat.rows * 4, cudaMemcpyDefault);
    if (e == cudaSuccess) e = cudaMemcpy(&st, d_status, 4, cudaMemcpyDeviceToHost);
  }
  cudaFree(d_units);
  cudaFree(d_x);
  cudaFree(d_y);
  cudaFree(d_part);
  cudaFree(d_cnt);
  cudaFree(d_status);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "matvec");
  if (st & ST_TIMEOUT) return set_err(nullptr, LLM_ERR_TIMEOUT, "a device-side wait exceeded its limit");
  return LLM_OK;
}

int llm_op_matvec(const llm_tensor* w, const float* x, float* y) { return op_matvec(w, x, y, false); }

int llm_op_matvec_w4a8(const llm_tensor* w, const float* x, float* y) { return op_matvec(w, x, y, true); }

}  // extern "C"

// ---- matvec without device allocation ---------------------------------------
// Scratch of llm_matvec_noalloc: split-row-tile partial sums, arrival
// counters and a status word, in one file-scope device array. Every GPU that
// loads this library holds it (4.2 MiB) until the process exits.
namespace {
constexpr size_t kNoAllocPartFloats = size_t(1) << 20;  // 4 MiB of partial sums
constexpr int kNoAllocCounters = 32768;                 // row tiles (32 rows each)
constexpr size_t kNoAllocBytes = kNoAllocPartFloats * 4 + (size_t)kNoAllocCounters * 4 + 256;
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

extern "C" int llm_matvec_noalloc(const llm_model* m, const char* name, const float* x, float* y,
                                  void* cuda_stream) {
  if (!m || !name || !x || !y) return set_err(nullptr, LLM_ERR_INVALID_ARG, "null argument");
  llm_model* mm = const_cast<llm_model*>(m);
  if (m->poisoned) return m->poisoned;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(mm, e, "cudaGetDevice");
  if (dev != m->device) return set_err(mm, LLM_ERR_INVALID_ARG, "the model's device must be the current device");
  if (dev >= kMaxDevices)
    return set_err(mm, LLM_ERR_UNSUPPORTED, "device ordinal " + std::to_string(dev) + " is beyond the " +
                                                std::to_string(kMaxDevices) + " devices this call serves");
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  {
    // the call reads its status back and synchronises: it cannot be captured
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_fail(mm, e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
      return set_err(mm, LLM_ERR_INVALID_ARG, "the stream is capturing: this call synchronises and cannot be captured");
  }
  if (!is_device_ptr(x) || !is_device_ptr(y)) return set_err(mm, LLM_ERR_INVALID_ARG, "x and y must be device memory");
  // the weight rows: a 4-bit tensor stored as a contiguous row range, or the tied bf16 LM head
  const Mat* mat = nullptr;
  int row0 = 0, rows = 0;
  const std::string nm(name);
  if (nm == "embed" && m->cfg.tied_embedding) {
    mat = &m->lm.m;
    rows = m->cfg.vocab;
  } else {
    auto it = m->places.find(nm);
    if (it == m->places.end() || it->second.kind != 0)
      return set_err(mm, LLM_ERR_NOT_FOUND, "no weight matrix " + nm + " stored as a contiguous row range");
    mat = &m->mats[it->second.mat];
    row0 = it->second.row0;
    rows = (int)m->shapes.at(nm).first;
  }
  Mat sub = *mat;
  sub.off = mat->off + (size_t)(row0 / 32) * mat->G * mat->unit_bytes();
  sub.rows = rows;
  sub.n_rt = (rows + 31) / 32;
  const GemvPlan g = plan_gemv(sub, m->n_sm);
  const size_t part_floats = (size_t)sub.n_rt * g.part.S * kTileRows;
  if (part_floats > kNoAllocPartFloats || sub.n_rt > kNoAllocCounters)
    return set_err(mm, LLM_ERR_UNSUPPORTED,
                   nm + " needs " + std::to_string(part_floats * 4 + sub.n_rt * 4) + " bytes of scratch; the static "
                   "scratch holds " + std::to_string(kNoAllocPartFloats * 4) + " bytes of partials and " +
                   std::to_string(kNoAllocCounters) + " row-tile counters");
  // one-time set-up on this device: the device address of the static array
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      e = cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_noalloc_scratch);
      if (e != cudaSuccess) {
        g_noalloc_ptr[dev] = nullptr;
        return cuda_fail(mm, e, "cudaGetSymbolAddress of the static scratch");
      }
    }
    base = g_noalloc_ptr[dev];
  }
  float* part = static_cast<float*>(base);
  int* counters = reinterpret_cast<int*>(static_cast<unsigned char*>(base) + kNoAllocPartFloats * 4);
  int* status = counters + kNoAllocCounters;
  // the array keeps the previous call's contents: counters and status must start at zero
  e = cudaMemsetAsync(counters, 0, (size_t)sub.n_rt * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, 4, st);
  if (e != cudaSuccess) return cuda_fail(mm, e, "scratch clear");
  GemvParams p{};
  p.units = m->d_arena + sub.off;
  p.n_rt = sub.n_rt;
  p.G = sub.G;
  p.K = sub.cols;
  p.rows = rows;
  p.unit_bytes = sub.unit_bytes();
  p.nslot = g.nslot;
  p.ring_bytes = g.ring;
  p.part = g.part;
  p.vec_mode = VEC_PLAIN;
  p.vin = x;
  p.epi = EPI_STORE;
  p.out = y;
  p.part_buf = part;
  p.counters = counters;
  p.status = status;
  // another model or call may have left the kernel's shared memory limit
  // below this matrix's need: raise it (never lower it)
  e = sub.bf16 ? raise_smem_limit(gemv_kernel<true>, g.smem) : raise_smem_limit(gemv_kernel<false>, g.smem);
  if (e != cudaSuccess) return cuda_fail(mm, e, "shared memory limit");
  e = sub.bf16 ? launch(gemv_kernel<true>, dim3(g.part.N), dim3(kGemvThreads), g.smem, st, false, p)
               : launch(gemv_kernel<false>, dim3(g.part.N), dim3(kGemvThreads), g.smem, st, false, p);
  int h_status = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h_status, status, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(mm, e, "matvec launch");
  if (h_status & ST_TIMEOUT) {
    mm->poisoned = LLM_ERR_TIMEOUT;
    return set_err(mm, LLM_ERR_TIMEOUT, "a device-side wait exceeded its limit");
  }
  return LLM_OK;
}
