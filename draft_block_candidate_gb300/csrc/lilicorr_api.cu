// The C ABI (include/lilicorr.h): weight validation and device arena, workspace planning,
// and the per-call sequence of kernels a1..a5 on the caller's stream.
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.cuh"

#ifndef LILICORR_PDL
#define LILICORR_PDL 1
#endif

namespace lilicorr {

// ---- bookkeeping
static std::atomic<uint64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed); }
static thread_local std::string t_last_error;
void set_last_error(const char* msg) { t_last_error = msg; }

// ---- per-device host state (one mutex: these are looked up once per launch at most)
static std::mutex g_dev_mu;
static std::map<std::pair<const void*, int>, int> g_smem_allowed;  // (kernel, device) -> bytes
static std::map<int, int> g_sm_count;                               // device -> SMs

static thread_local bool t_pdl = false;
bool pdl_enabled() { return t_pdl; }
PdlScope::PdlScope(bool on) : prev(t_pdl) { t_pdl = on; }
PdlScope::~PdlScope() { t_pdl = prev; }
void PdlScope::set(bool on) { t_pdl = on; }

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  auto it = g_sm_count.find(dev);
  if (it != g_sm_count.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  g_sm_count[dev] = n;
  return n;
}

cudaError_t allow_dynamic_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  int& have = g_smem_allowed[{kernel, dev}];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

static lilicorr_status cuda_fail(cudaError_t e, const char* where) {
  t_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return LILICORR_ERR_CUDA;
}
#define LC_CUDA(expr, where)                        \
  do {                                              \
    cudaError_t e_ = (expr);                        \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

// ---- per-kernel timing: events recorded on the caller's stream after each launch
enum Slot : int {
  T_LOGIT = 0, T_CONF, T_NODE, T_NORM, T_QKV, T_ATTN, T_OUT, T_FFN1, T_FFN2, T_TARGET, T_FUSE,
  T_HEADS, T_SCORES, T_WALK, NSLOT
};
static const char* kSlotNames[NSLOT] = {
    "logit_pass", "conf_hidden", "node_gemm", "rmsnorm", "qkv_gemm", "attention", "out_gemm",
    "ffn1_gemm", "ffn2_gemm", "target_terms", "fuse_gemm", "heads_gemm", "pair_scores",
    "greedy_walk"};

struct CallRecord {
  cudaEvent_t start;
  std::vector<std::pair<int, cudaEvent_t>> marks;
};
struct StageTimer {
  std::mutex mu;
  bool enabled = false;
  std::vector<CallRecord> pending;
  double ms[NSLOT] = {};
  int64_t launches[NSLOT] = {};
  int64_t calls = 0;
};
static StageTimer g_timer;

struct CallTimer {
  bool on = false;
  cudaStream_t stream = nullptr;
  CallRecord rec{};
  cudaError_t begin(cudaStream_t s) {
    {
      std::lock_guard<std::mutex> lk(g_timer.mu);
      on = g_timer.enabled;
    }
    stream = s;
    if (!on) return cudaSuccess;
    cudaError_t e = cudaEventCreate(&rec.start);
    return e == cudaSuccess ? cudaEventRecord(rec.start, s) : e;
  }
  cudaError_t mark(int slot) {
    if (!on) return cudaSuccess;
    cudaEvent_t e;
    cudaError_t r = cudaEventCreate(&e);
    if (r != cudaSuccess) return r;
    rec.marks.push_back({slot, e});
    return cudaEventRecord(e, stream);
  }
  void finish() {
    if (!on) return;
    std::lock_guard<std::mutex> lk(g_timer.mu);
    g_timer.pending.push_back(rec);
  }
};

}  // namespace lilicorr

using namespace lilicorr;

struct lilicorr_weights {
  lilicorr_dims d;
  int device;
  void* arena;
  // bf16 (tensor-core operands and the gathered embedding)
  // fuse_w is [Wh | Wt | Wht] ([H, 3H]); fuse_w2 = [Wh | Wht] ([H, 2H]) for the
  // contraction over [h, h*t]; the Wt t term is a per-block bias
  const __nv_bfloat16 *embed, *conf_w2, *fuse_w, *fuse_w2, *heads_w, *anchor_w, *tgt_w;
  // f32 (exact widening of the bf16 inputs)
  const float *slot_table, *rank_table, *conf_w1, *conf_b1, *conf_b2, *fuse_b, *heads_b, *anchor_b,
      *tgt_b;
  struct Layer {
    const __nv_bfloat16 *in_w, *out_w, *w1, *w2;
    const float *norm1, *in_b, *out_b, *dist, *same, *norm2, *b1, *b2;
  };
  std::vector<Layer> layers;
};

namespace {

struct Expect {
  std::vector<int64_t> shape;
  bool f32;  // widened to f32 in the arena
};

std::map<std::string, Expect> expected_tensors(const lilicorr_dims& d) {
  const int64_t H = d.hidden, F = d.ffn, E = d.d_e, nh = d.heads, Bm = d.B_max, Km = d.K_max;
  std::map<std::string, Expect> m;
  m["embed"] = {{d.V, H}, false};
  m["slot_table"] = {{Bm - 1, H}, true};
  m["rank_table"] = {{Km, H}, true};
  m["conf.w1"] = {{H, 5}, true};
  m["conf.b1"] = {{H}, true};
  m["conf.w2"] = {{H, H}, false};
  m["conf.b2"] = {{H}, true};
  for (int l = 0; l < d.layers; ++l) {
    const std::string p = "layers." + std::to_string(l) + ".";
    m[p + "norm1"] = {{H}, true};
    m[p + "in_proj_w"] = {{3 * H, H}, false};
    m[p + "in_proj_b"] = {{3 * H}, true};
    m[p + "out_proj_w"] = {{H, H}, false};
    m[p + "out_proj_b"] = {{H}, true};
    m[p + "dist_bias"] = {{nh, 2 * Bm - 3}, true};
    m[p + "same_bias"] = {{nh}, true};
    m[p + "norm2"] = {{H}, true};
    m[p + "ffn.w1"] = {{F, H}, false};
    m[p + "ffn.b1"] = {{F}, true};
    m[p + "ffn.w2"] = {{H, F}, false};
    m[p + "ffn.b2"] = {{H}, true};
  }
  m["fuse.w"] = {{H, 3 * H}, false};
  m["fuse.b"] = {{H}, true};
  m["head_out.w"] = {{E, H}, false};
  m["head_out.b"] = {{E}, true};
  m["head_in.w"] = {{E, H}, false};
  m["head_in.b"] = {{E}, true};
  m["head_anchor.w"] = {{E, H}, false};
  m["head_anchor.b"] = {{E}, true};
  return m;
}

bool dims_ok(const lilicorr_dims& d) {
  if (d.layers < 0 || d.layers > 64) return false;
  if (d.hidden <= 0 || d.hidden % 64 != 0 || d.hidden > 4096) return false;
  if (d.heads <= 0 || d.hidden % d.heads != 0) return false;
  const int dh = d.hidden / d.heads;
  if (dh != 32 && dh != 64 && dh != 128) return false;
  if (d.ffn <= 0 || d.ffn % 64 != 0) return false;
  if (d.d_e <= 0 || d.d_e % 32 != 0 || d.d_e > 256) return false;
  if (d.B_max < 2 || d.B_max > 64) return false;
  if (d.K_max < 1 || d.K_max > 32) return false;
  if (d.V < 1 || d.V > (int64_t(1) << 31) - 2) return false;
  if (!(d.sigma == d.sigma) || !(d.rms_eps >= 0.f)) return false;
  return true;
}

float bf16_to_f32(uint16_t b) {
  uint32_t u = uint32_t(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace layout of one rerank call.
struct WsPlan {
  size_t k1, cand_id, cand_logit, lse, act1, X, qkv, ffh, heads, scores, tgt, total;
};

WsPlan ws_plan(const lilicorr_dims& d, int64_t batch, int B, int K, int esize) {
  WsPlan p{};
  const int64_t rows = batch * (B - 1);
  const int64_t M = rows * K;
  const int64_t H = d.hidden, F = d.ffn, E = d.d_e;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  p.k1 = take(k1_workspace_bytes(batch, B, d.V, esize));
  p.cand_id = take(size_t(M) * 4);
  p.cand_logit = take(size_t(M) * 4);
  p.lse = take(size_t(rows) * 4);
  p.act1 = take(size_t(M) * 2 * H * 2);
  p.X = take(size_t(M) * H * 4);
  p.qkv = take(size_t(M) * 6 * H * 2);
  p.ffh = take(size_t(M) * 2 * F * 2);
  p.heads = take(size_t(M) * 2 * E * 4);
  p.scores = take(size_t(rows) * K * K * 4);
  p.tgt = take(size_t(batch) * (H + E) * 4);
  p.total = off;
  return p;
}

lilicorr_status check_call(const lilicorr_weights* w, lilicorr_dtype ldtype, int64_t batch,
                           int32_t B, int64_t V, int32_t K) {
  if (!w) return LILICORR_ERR_INVALID_ARG;
  if (ldtype != LILICORR_F32 && ldtype != LILICORR_BF16) return LILICORR_ERR_INVALID_ARG;
  if (batch < 1 || B < 2 || B > w->d.B_max || V != w->d.V) return LILICORR_ERR_INVALID_ARG;
  if (K < 1 || K > w->d.K_max || K > V) return LILICORR_ERR_INVALID_ARG;
  if (batch * (B - 1) * int64_t(K) > (int64_t(1) << 31) - 1) return LILICORR_ERR_INVALID_ARG;
  if (V * (ldtype == LILICORR_BF16 ? 2 : 4) > (int64_t(1) << 31) - 64) return LILICORR_ERR_INVALID_ARG;
  return LILICORR_OK;
}

}  // namespace

extern "C" {

const char* lilicorr_status_string(lilicorr_status s) {
  switch (s) {
    case LILICORR_OK: return "ok";
    case LILICORR_ERR_INVALID_ARG: return "invalid argument";
    case LILICORR_ERR_UNSUPPORTED: return "unsupported";
    case LILICORR_ERR_WEIGHTS_MISSING: return "head tensor missing";
    case LILICORR_ERR_WEIGHTS_SURPLUS: return "unknown head tensor";
    case LILICORR_ERR_WEIGHTS_SHAPE: return "head tensor shape or dtype mismatch";
    case LILICORR_ERR_CUDA: return "CUDA error";
    case LILICORR_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case LILICORR_ERR_DEVICE: return "device-side error";
  }
  return "unknown status";
}

const char* lilicorr_last_error(void) { return t_last_error.c_str(); }

uint64_t lilicorr_launch_count(void) { return g_launches.load(); }

lilicorr_status lilicorr_device_error(uint32_t* code) {
  if (!code) return LILICORR_ERR_INVALID_ARG;
  *code = 0;
  LC_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  LC_CUDA(k1_read_device_error(code), "read device error");
  LC_CUDA(tc_read_device_error(code), "read device error");
  LC_CUDA(at_read_device_error(code), "read device error");
  return *code ? LILICORR_ERR_DEVICE : LILICORR_OK;
}

lilicorr_status lilicorr_weights_create(const lilicorr_dims* dims, const lilicorr_tensor* tensors,
                                        int32_t n, int device, lilicorr_weights** out) {
  if (!dims || !out || (n > 0 && !tensors) || n < 0) return LILICORR_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims_ok(*dims)) return LILICORR_ERR_INVALID_ARG;
  const auto exp = expected_tensors(*dims);
  std::map<std::string, const lilicorr_tensor*> given;
  for (int i = 0; i < n; ++i) {
    if (!tensors[i].name) return LILICORR_ERR_INVALID_ARG;
    const std::string nm(tensors[i].name);
    if (!exp.count(nm)) return LILICORR_ERR_WEIGHTS_SURPLUS;
    if (given.count(nm)) return LILICORR_ERR_INVALID_ARG;
    given[nm] = &tensors[i];
  }
  for (const auto& kv : exp)
    if (!given.count(kv.first)) return LILICORR_ERR_WEIGHTS_MISSING;
  for (const auto& kv : exp) {
    const lilicorr_tensor* t = given[kv.first];
    if (t->dtype != LILICORR_BF16) return LILICORR_ERR_WEIGHTS_SHAPE;
    if (t->ndim != int32_t(kv.second.shape.size())) return LILICORR_ERR_WEIGHTS_SHAPE;
    for (int i = 0; i < t->ndim; ++i)
      if (t->shape[i] != kv.second.shape[i]) return LILICORR_ERR_WEIGHTS_SHAPE;
    if (!t->host_data) return LILICORR_ERR_INVALID_ARG;
  }

  // Host image of the arena.
  std::vector<uint8_t> img;
  std::map<std::string, size_t> off;
  auto numel = [](const std::vector<int64_t>& s) {
    int64_t k = 1;
    for (auto v : s) k *= v;
    return k;
  };
  auto put_bf16 = [&](const std::string& name, const void* src, int64_t cnt) {
    const size_t o = align256(img.size());
    img.resize(o + size_t(cnt) * 2);
    std::memcpy(img.data() + o, src, size_t(cnt) * 2);
    off[name] = o;
  };
  auto put_f32 = [&](const std::string& name, const void* src, int64_t cnt) {
    const size_t o = align256(img.size());
    img.resize(o + size_t(cnt) * 4);
    const uint16_t* s = static_cast<const uint16_t*>(src);
    float* d = reinterpret_cast<float*>(img.data() + o);
    for (int64_t i = 0; i < cnt; ++i) d[i] = bf16_to_f32(s[i]);
    off[name] = o;
  };
  for (const auto& kv : exp) {
    if (kv.first == "head_out.w" || kv.first == "head_in.w" || kv.first == "head_out.b" ||
        kv.first == "head_in.b")
      continue;
    const int64_t cnt = numel(kv.second.shape);
    if (kv.second.f32)
      put_f32(kv.first, given[kv.first]->host_data, cnt);
    else
      put_bf16(kv.first, given[kv.first]->host_data, cnt);
  }
  // fusion weight without its target-state block: [Wh | Wht] [H, 2H]
  {
    const int64_t H = dims->hidden;
    const size_t o = align256(img.size());
    img.resize(o + size_t(2 * H * H) * 2);
    const uint8_t* src = static_cast<const uint8_t*>(given["fuse.w"]->host_data);
    for (int64_t n = 0; n < H; ++n) {
      std::memcpy(img.data() + o + size_t(n * 2 * H) * 2, src + size_t(n * 3 * H) * 2, size_t(H) * 2);
      std::memcpy(img.data() + o + size_t(n * 2 * H + H) * 2, src + size_t(n * 3 * H + 2 * H) * 2,
                  size_t(H) * 2);
    }
    off["fuse.w2"] = o;
  }
  // out and in heads are one contraction: W = [Wout; Win] [2E, H], b = [bout; bin].
  {
    const int64_t EH = int64_t(dims->d_e) * dims->hidden;
    const size_t o = align256(img.size());
    img.resize(o + size_t(2 * EH) * 2);
    std::memcpy(img.data() + o, given["head_out.w"]->host_data, size_t(EH) * 2);
    std::memcpy(img.data() + o + size_t(EH) * 2, given["head_in.w"]->host_data, size_t(EH) * 2);
    off["heads.w"] = o;
    const size_t ob = align256(img.size());
    img.resize(ob + size_t(2 * dims->d_e) * 4);
    float* d = reinterpret_cast<float*>(img.data() + ob);
    const uint16_t* so = static_cast<const uint16_t*>(given["head_out.b"]->host_data);
    const uint16_t* si = static_cast<const uint16_t*>(given["head_in.b"]->host_data);
    for (int e = 0; e < dims->d_e; ++e) {
      d[e] = bf16_to_f32(so[e]);
      d[dims->d_e + e] = bf16_to_f32(si[e]);
    }
    off["heads.b"] = ob;
  }
  // the two per-block terms of the target state are one contraction:
  // [Wt; Wa] [H + E, H] (Wt = the middle H columns of fuse.w), b = [bf; ba]
  {
    const int64_t H = dims->hidden, E = dims->d_e;
    const size_t o = align256(img.size());
    img.resize(o + size_t((H + E) * H) * 2);
    const uint8_t* fw = static_cast<const uint8_t*>(given["fuse.w"]->host_data);
    for (int64_t n = 0; n < H; ++n)
      std::memcpy(img.data() + o + size_t(n * H) * 2, fw + size_t(n * 3 * H + H) * 2, size_t(H) * 2);
    std::memcpy(img.data() + o + size_t(H * H) * 2, given["head_anchor.w"]->host_data,
                size_t(E * H) * 2);
    off["tgt.w"] = o;
    const size_t ob = align256(img.size());
    img.resize(ob + size_t(H + E) * 4);
    float* d = reinterpret_cast<float*>(img.data() + ob);
    const uint16_t* fb = static_cast<const uint16_t*>(given["fuse.b"]->host_data);
    const uint16_t* ab = static_cast<const uint16_t*>(given["head_anchor.b"]->host_data);
    for (int64_t n = 0; n < H; ++n) d[n] = bf16_to_f32(fb[n]);
    for (int64_t e = 0; e < E; ++e) d[H + e] = bf16_to_f32(ab[e]);
    off["tgt.b"] = ob;
  }

  int prev = 0;
  LC_CUDA(cudaGetDevice(&prev), "cudaGetDevice");
  LC_CUDA(cudaSetDevice(device), "cudaSetDevice");
  void* arena = nullptr;
  cudaError_t e = cudaMalloc(&arena, img.size());
  if (e == cudaSuccess) e = cudaMemcpy(arena, img.data(), img.size(), cudaMemcpyHostToDevice);
  cudaSetDevice(prev);
  if (e != cudaSuccess) {
    if (arena) cudaFree(arena);
    return cuda_fail(e, "weights arena");
  }

  auto* w = new lilicorr_weights();
  w->d = *dims;
  w->device = device;
  w->arena = arena;
  auto bf = [&](const std::string& nm) {
    return reinterpret_cast<const __nv_bfloat16*>(static_cast<uint8_t*>(arena) + off.at(nm));
  };
  auto f32 = [&](const std::string& nm) {
    return reinterpret_cast<const float*>(static_cast<uint8_t*>(arena) + off.at(nm));
  };
  w->embed = bf("embed");
  w->conf_w2 = bf("conf.w2");
  w->fuse_w = bf("fuse.w");
  w->fuse_w2 = bf("fuse.w2");
  w->heads_w = bf("heads.w");
  w->anchor_w = bf("head_anchor.w");
  w->tgt_w = bf("tgt.w");
  w->slot_table = f32("slot_table");
  w->rank_table = f32("rank_table");
  w->conf_w1 = f32("conf.w1");
  w->conf_b1 = f32("conf.b1");
  w->conf_b2 = f32("conf.b2");
  w->fuse_b = f32("fuse.b");
  w->heads_b = f32("heads.b");
  w->anchor_b = f32("head_anchor.b");
  w->tgt_b = f32("tgt.b");
  for (int l = 0; l < dims->layers; ++l) {
    const std::string p = "layers." + std::to_string(l) + ".";
    lilicorr_weights::Layer L;
    L.in_w = bf(p + "in_proj_w");
    L.out_w = bf(p + "out_proj_w");
    L.w1 = bf(p + "ffn.w1");
    L.w2 = bf(p + "ffn.w2");
    L.norm1 = f32(p + "norm1");
    L.in_b = f32(p + "in_proj_b");
    L.out_b = f32(p + "out_proj_b");
    L.dist = f32(p + "dist_bias");
    L.same = f32(p + "same_bias");
    L.norm2 = f32(p + "norm2");
    L.b1 = f32(p + "ffn.b1");
    L.b2 = f32(p + "ffn.b2");
    w->layers.push_back(L);
  }
  *out = w;
  return LILICORR_OK;
}

void lilicorr_weights_destroy(lilicorr_weights* w) {
  if (!w) return;
  if (w->arena) cudaFree(w->arena);
  delete w;
}

lilicorr_status lilicorr_weights_dims(const lilicorr_weights* w, lilicorr_dims* out) {
  if (!w || !out) return LILICORR_ERR_INVALID_ARG;
  *out = w->d;
  return LILICORR_OK;
}

size_t lilicorr_workspace_bytes(const lilicorr_weights* w, int64_t batch, int32_t B, int32_t K) {
  if (check_call(w, LILICORR_BF16, batch, B, w ? w->d.V : 0, K) != LILICORR_OK) return 0;
  // the logit-pass partials are sized for the larger element (f32 rows are longer)
  const WsPlan a = ws_plan(w->d, batch, B, K, 2), b = ws_plan(w->d, batch, B, K, 4);
  return (a.total > b.total ? a.total : b.total) + 256;
}

size_t lilicorr_topk_lse_workspace_bytes(int64_t batch, int32_t B, int64_t V, int32_t K,
                                         lilicorr_dtype ldtype) {
  if (batch < 1 || B < 2 || V < 1 || K < 1 || K > 32 || K > V) return 0;
  if (ldtype != LILICORR_F32 && ldtype != LILICORR_BF16) return 0;
  return k1_workspace_bytes(batch, B, V, ldtype == LILICORR_BF16 ? 2 : 4);
}

lilicorr_status lilicorr_topk_lse(const void* logits, lilicorr_dtype ldtype, int64_t batch,
                                  int32_t B, int64_t V, int32_t K, int32_t* cand_id,
                                  float* cand_logit, float* lse, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (!logits || !cand_id || !cand_logit || !lse) return LILICORR_ERR_INVALID_ARG;
  if (batch < 1 || B < 2 || V < 1 || V > (int64_t(1) << 31) - 2 || K < 1 || K > 32 || K > V)
    return LILICORR_ERR_INVALID_ARG;
  if (ldtype != LILICORR_F32 && ldtype != LILICORR_BF16) return LILICORR_ERR_INVALID_ARG;
  const int es = ldtype == LILICORR_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % es) return LILICORR_ERR_INVALID_ARG;
  if (V * es > (int64_t(1) << 31) - 64) return LILICORR_ERR_INVALID_ARG;  // row < 2 GiB
  const size_t need = k1_workspace_bytes(batch, B, V, es);
  if (need && (!workspace || workspace_bytes < need ||
               reinterpret_cast<uintptr_t>(workspace) % 256))
    return LILICORR_ERR_WORKSPACE;
  LC_CUDA(k1_launch(logits, es, batch, B, V, K, cand_id, cand_logit, lse, workspace,
                    static_cast<cudaStream_t>(stream)),
          "logit pass");
  return LILICORR_OK;
}

size_t lilicorr_topk_lse_shard_record_bytes(int32_t K) {
  return (K < 1 || K > 32) ? 0 : k1_shard_record_bytes(K);
}

lilicorr_status lilicorr_topk_lse_shard(const void* logits, lilicorr_dtype ldtype,
                                        int64_t batch, int32_t B, int64_t V_shard,
                                        int64_t row_stride, int64_t id_offset, int32_t K,
                                        void* records, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  if (!logits || !records) return LILICORR_ERR_INVALID_ARG;
  if (batch < 1 || B < 2 || V_shard < 1 || K < 1 || K > 32) return LILICORR_ERR_INVALID_ARG;
  if (row_stride < V_shard || id_offset < 0 || id_offset + V_shard > (int64_t(1) << 31) - 2)
    return LILICORR_ERR_INVALID_ARG;
  if (ldtype != LILICORR_F32 && ldtype != LILICORR_BF16) return LILICORR_ERR_INVALID_ARG;
  const int es = ldtype == LILICORR_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % es || reinterpret_cast<uintptr_t>(records) % 4)
    return LILICORR_ERR_INVALID_ARG;
  if (V_shard * es > (int64_t(1) << 31) - 64) return LILICORR_ERR_INVALID_ARG;
  const size_t need = k1_workspace_bytes(batch, B, V_shard, es);
  if (need && (!workspace || workspace_bytes < need ||
               reinterpret_cast<uintptr_t>(workspace) % 256))
    return LILICORR_ERR_WORKSPACE;
  LC_CUDA(k1_launch(logits, es, batch, B, V_shard, K, nullptr, nullptr, nullptr, workspace,
                    static_cast<cudaStream_t>(stream), row_stride, static_cast<int>(id_offset),
                    records),
          "logit pass (vocabulary shard)");
  return LILICORR_OK;
}

lilicorr_status lilicorr_topk_lse_merge(const void* records, int32_t n_shards, int64_t rows,
                                        int32_t K, int32_t* cand_id, float* cand_logit,
                                        float* lse, void* stream) {
  if (!records || !cand_id || !cand_logit || !lse) return LILICORR_ERR_INVALID_ARG;
  if (n_shards < 1 || rows < 1 || K < 1 || K > 32 || reinterpret_cast<uintptr_t>(records) % 4)
    return LILICORR_ERR_INVALID_ARG;
  LC_CUDA(k1_merge_launch(records, n_shards, rows, K, cand_id, cand_logit, lse,
                          static_cast<cudaStream_t>(stream)),
          "shard merge");
  return LILICORR_OK;
}

size_t lilicorr_lm_head_workspace_bytes(int64_t rows, int64_t V, int32_t D, int32_t K) {
  if (!lm_head_supported(rows, V, D, K)) return 0;
  return align256(lm_head_records_bytes(rows, V, K));
}

lilicorr_status lilicorr_lm_head_topk_lse(const void* hidden, const void* w_lm, int64_t rows,
                                          int64_t V, int32_t D, int32_t K, int32_t* cand_id,
                                          float* cand_logit, float* lse, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (!hidden || !w_lm || !cand_id || !cand_logit || !lse) return LILICORR_ERR_INVALID_ARG;
  if (!lm_head_supported(rows, V, D, K)) return LILICORR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(hidden) % 16 || reinterpret_cast<uintptr_t>(w_lm) % 16)
    return LILICORR_ERR_INVALID_ARG;
  const size_t need = lilicorr_lm_head_workspace_bytes(rows, V, D, K);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return LILICORR_ERR_WORKSPACE;
  LC_CUDA(launch_lm_head_topk(static_cast<const __nv_bfloat16*>(hidden),
                              static_cast<const __nv_bfloat16*>(w_lm), rows, V, D, K, workspace,
                              cand_id, cand_logit, lse, static_cast<cudaStream_t>(stream)),
          "lm head + top-k / lse");
  return LILICORR_OK;
}

lilicorr_status lilicorr_greedy_walk(const float* pair_scores, const int32_t* cand_id,
                                     const int32_t* anchor_ids, int64_t batch, int32_t B,
                                     int32_t K, int32_t* tokens, int32_t* choice,
                                     float* path_score, void* stream) {
  if (!pair_scores || !cand_id || !tokens) return LILICORR_ERR_INVALID_ARG;
  if (batch < 1 || B < 2 || B > 64 || K < 1 || K > 32) return LILICORR_ERR_INVALID_ARG;
  LC_CUDA(launch_greedy_walk(pair_scores, cand_id, anchor_ids, batch, B, K, tokens, choice,
                             path_score, static_cast<cudaStream_t>(stream)),
          "greedy walk");
  return LILICORR_OK;
}

lilicorr_status lilicorr_viterbi(const float* pair_scores, const int32_t* cand_id,
                                 const int32_t* anchor_ids, int64_t batch, int32_t B, int32_t K,
                                 int32_t* tokens, int32_t* choice, float* path_score,
                                 double* total, void* stream) {
  if (!pair_scores || !cand_id || !tokens) return LILICORR_ERR_INVALID_ARG;
  if (batch < 1 || B < 2 || B > 64 || K < 1 || K > 32) return LILICORR_ERR_INVALID_ARG;
  LC_CUDA(launch_viterbi(pair_scores, cand_id, anchor_ids, batch, B, K, tokens, choice,
                         path_score, total, static_cast<cudaStream_t>(stream)),
          "viterbi");
  return LILICORR_OK;
}

lilicorr_status lilicorr_sample_walk(const float* pair_scores, const int32_t* cand_id,
                                     const int32_t* anchor_ids, const float* temperature,
                                     const float* uniforms, int64_t batch, int32_t B,
                                     int32_t K, int32_t* tokens, int32_t* choice,
                                     float* path_score, float* proposal, void* stream) {
  if (!pair_scores || !cand_id || !tokens) return LILICORR_ERR_INVALID_ARG;
  if (temperature && !uniforms) return LILICORR_ERR_INVALID_ARG;
  if (batch < 1 || B < 2 || K < 1 || K > 32) return LILICORR_ERR_INVALID_ARG;
  LC_CUDA(launch_sample_walk(pair_scores, cand_id, anchor_ids, temperature, uniforms, batch, B,
                             K, tokens, choice, path_score, proposal,
                             static_cast<cudaStream_t>(stream)),
          "sample walk");
  return LILICORR_OK;
}

lilicorr_status lilicorr_rerank(const lilicorr_weights* w, const void* logits,
                                lilicorr_dtype ldtype, int64_t batch, int32_t B, int64_t V,
                                int32_t K, const void* slot_hidden, const void* target_state,
                                const int32_t* anchor_ids, int32_t* tokens, float* path_score,
                                const lilicorr_taps* taps, void* workspace,
                                size_t workspace_bytes, void* stream_) {
  lilicorr_status st = check_call(w, ldtype, batch, B, V, K);
  if (st != LILICORR_OK) return st;
  if (!logits || !tokens || !path_score) return LILICORR_ERR_INVALID_ARG;
  const int es = ldtype == LILICORR_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % es) return LILICORR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(slot_hidden) % 16 || reinterpret_cast<uintptr_t>(target_state) % 16)
  {
    lilicorr::set_last_error("slot_hidden / target_state must be 16-byte aligned");
    return LILICORR_ERR_INVALID_ARG;
  }
  const WsPlan pl = ws_plan(w->d, batch, B, K, es);
  if (!workspace || workspace_bytes < pl.total || reinterpret_cast<uintptr_t>(workspace) % 256)
    return LILICORR_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const lilicorr_taps none{};
  const lilicorr_taps& tp = taps ? *taps : none;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const lilicorr_dims& d = w->d;
  const int H = d.hidden, F = d.ffn, E = d.d_e;
  const int S = (B - 1) * K;
  const int64_t M = batch * S;

  int32_t* cand_id = tp.cand_id ? tp.cand_id : reinterpret_cast<int32_t*>(ws + pl.cand_id);
  float* cand_logit = tp.cand_logit ? tp.cand_logit : reinterpret_cast<float*>(ws + pl.cand_logit);
  float* lse = tp.lse ? tp.lse : reinterpret_cast<float*>(ws + pl.lse);
  float* scores = tp.pair_scores ? tp.pair_scores : reinterpret_cast<float*>(ws + pl.scores);
  __nv_bfloat16* act1 = reinterpret_cast<__nv_bfloat16*>(ws + pl.act1);
  float* X = reinterpret_cast<float*>(ws + pl.X);
  __nv_bfloat16* qkv = reinterpret_cast<__nv_bfloat16*>(ws + pl.qkv);
  __nv_bfloat16* ffh = reinterpret_cast<__nv_bfloat16*>(ws + pl.ffh);
  float* heads = reinterpret_cast<float*>(ws + pl.heads);
  const __nv_bfloat16* target = static_cast<const __nv_bfloat16*>(target_state);

  CallTimer tm;
  LC_CUDA(tm.begin(stream), "timing event");
#define MARK(slot) LC_CUDA(tm.mark(slot), "timing event")
  // Up to 32,768 lattice tokens, kernels after the first are launched as programmatic
  // dependents of the one before (each waits for its predecessor in pdl_wait before
  // touching memory), so that a launch and its set-up overlap the previous kernel: about
  // 10 us per call at one to 64 blocks (single request 187 -> 177 us).  Larger batches
  // keep plain launches (batch 256: 1,084 against 1,090 us with them).  The first kernel
  // follows whatever the stream held before the call, and a kernel after a copy follows
  // the copy.
  const bool use_pdl = LILICORR_PDL != 0 && M <= 32768;
  PdlScope pdl(false);
  // a1: logit pass
  LC_CUDA(k1_launch(logits, es, batch, B, V, K, cand_id, cand_logit, lse, ws + pl.k1, stream),
          "logit pass");
  MARK(T_LOGIT);
  pdl.set(use_pdl);
  // a2: node build.  The confidence layer's hidden units are made inside the node GEMM
  // from each candidate's five features, except at hidden width 256, where the
  // standalone layer (weights in shared memory) and a TMA-fed node GEMM measured faster
  // (81 against 91 us per step at batch 256; the node GEMM is bound by its gather
  // epilogue, which the producer warps slow down; at width 512 the in-kernel form saves
  // 17 us)
  const bool conf_apart = H == 256;
  if (conf_apart) {
    LC_CUDA(launch_conf_hidden(cand_logit, lse, M, K, H, w->conf_w1, w->conf_b1, act1, stream),
            "confidence features");
    MARK(T_CONF);
  }
  {
    GemmArgs g{};
    if (conf_apart) {
      g.A = act1;
    } else {
      g.asrc = ASRC_CONF; g.a_cl = cand_logit; g.a_lse = lse; g.a_w1 = w->conf_w1;
      g.a_b1 = w->conf_b1;
    }
    g.W = w->conf_w2; g.M = M; g.N = H; g.Kw = H; g.Ka = 2 * H; g.bias = w->conf_b2;
    g.out = X; g.embed = w->embed; g.cand_id = cand_id; g.slot_table = w->slot_table;
    g.rank_table = w->rank_table; g.slot_hidden = static_cast<const __nv_bfloat16*>(slot_hidden);
    g.K = K; g.B = B; g.vocab = d.V; g.nodes_tap = tp.nodes;
    LC_CUDA(launch_gemm(EPI_NODE, g, stream), "node gemm");
    MARK(T_NODE);
  }
  // a3: encoder
  for (const auto& L : w->layers) {
    LC_CUDA(launch_rmsnorm_split(X, L.norm1, M, H, d.rms_eps, act1, stream), "rmsnorm");
    MARK(T_NORM);
    GemmArgs g{};
    g.A = act1; g.W = L.in_w; g.M = M; g.N = 3 * H; g.Kw = H; g.Ka = 2 * H; g.bias = L.in_b;
    g.out_split = qkv;
    LC_CUDA(launch_gemm(EPI_SPLIT, g, stream), "qkv gemm");
    MARK(T_QKV);
    if (attention_tc_supported(S, K, H, d.heads, d.B_max))
      LC_CUDA(launch_attention_tc(qkv, batch, S, K, H, d.heads, d.B_max, L.dist, L.same, act1,
                                  stream),
              "attention");
    else if (attention_tc_long_supported(S, K, H, d.heads, d.B_max))
      LC_CUDA(launch_attention_tc_long(qkv, batch, S, K, H, d.heads, d.B_max, L.dist, L.same,
                                       act1, stream),
              "attention");
    else
      LC_CUDA(launch_attention(qkv, batch, S, K, H, d.heads, d.B_max, L.dist, L.same, act1, stream),
              "attention");
    MARK(T_ATTN);
    g = GemmArgs{};
    g.A = act1; g.W = L.out_w; g.M = M; g.N = H; g.Kw = H; g.Ka = 2 * H; g.bias = L.out_b; g.out = X;
    LC_CUDA(launch_gemm(EPI_RESID, g, stream), "out-proj gemm");
    MARK(T_OUT);
    LC_CUDA(launch_rmsnorm_split(X, L.norm2, M, H, d.rms_eps, act1, stream), "rmsnorm");
    MARK(T_NORM);
    g = GemmArgs{};
    g.A = act1; g.W = L.w1; g.M = M; g.N = F; g.Kw = H; g.Ka = 2 * H; g.bias = L.b1; g.out_split = ffh;
    LC_CUDA(launch_gemm(EPI_SPLIT_SILU, g, stream), "ffn1 gemm");
    MARK(T_FFN1);
    g = GemmArgs{};
    g.A = ffh; g.W = L.w2; g.M = M; g.N = H; g.Kw = F; g.Ka = 2 * F; g.bias = L.b2; g.out = X;
    LC_CUDA(launch_gemm(EPI_RESID, g, stream), "ffn2 gemm");
    MARK(T_FFN2);
  }
  if (tp.hidden) {
    LC_CUDA(cudaMemcpyAsync(tp.hidden, X, size_t(M) * H * 4, cudaMemcpyDeviceToDevice, stream),
            "hidden tap");
    pdl.set(false);
  }
  // a4: fusion and heads
  // per-block target terms [Wt t + bf | Wa t + ba], one row per block
  float* tgt = reinterpret_cast<float*>(ws + pl.tgt);
  const int HE = static_cast<int>(H + E);
  if (target) {
    GemmArgs g{};
    g.A = target; g.W = w->tgt_w; g.M = batch; g.N = HE; g.Kw = H; g.Ka = H; g.bias = w->tgt_b;
    g.out = tgt;
    LC_CUDA(launch_gemm(EPI_F32, g, stream), "target terms gemm");
  } else {
    LC_CUDA(launch_rows_bias(w->tgt_b, batch, HE, tgt, stream), "target terms");
  }
  MARK(T_TARGET);
  pdl.set(use_pdl);
  {
    // SiLU(Wh h + Wht (h*t) + [Wt t + bf]_block): A = [h, h*t] split, made inside the GEMM
    // from the residual stream and the block's target state; bias per block
    GemmArgs g{};
    g.asrc = ASRC_FUSION; g.a_x = X; g.a_t = target; g.a_group = S;
    g.W = w->fuse_w2; g.M = M; g.N = H; g.Kw = 2 * H; g.Ka = 4 * H; g.bias = tgt;
    g.bias_group = S; g.bias_stride = HE; g.out_split = act1;
    LC_CUDA(launch_gemm(EPI_SPLIT_SILU, g, stream), "fusion gemm");
    MARK(T_FUSE);
    g = GemmArgs{};
    g.A = act1; g.W = w->heads_w; g.M = M; g.N = 2 * E; g.Kw = H; g.Ka = 2 * H; g.bias = w->heads_b;
    g.out = heads;
    LC_CUDA(launch_gemm(EPI_F32, g, stream), "heads gemm");
    MARK(T_HEADS);
  }
  // a4 scores (with the anchor head) + a5 walk
  LC_CUDA(launch_pair_scores(heads, tgt + H, HE, batch, B, K, E, d.sigma, scores, tp.out_vec,
                             tp.in_vec, tp.anchor_vec, stream),
          "pair scores");
  MARK(T_SCORES);
  LC_CUDA(launch_greedy_walk(scores, cand_id, anchor_ids, batch, B, K, tokens, tp.choice,
                             path_score, stream),
          "greedy walk");
  MARK(T_WALK);
#undef MARK
  tm.finish();
  return LILICORR_OK;
}

size_t lilicorr_workspace_bytes_host(const lilicorr_weights* w, int64_t batch, int32_t B,
                                     int32_t K, lilicorr_dtype ldtype) {
  const size_t base = lilicorr_workspace_bytes(w, batch, B, K);
  if (!base) return 0;
  const int es = ldtype == LILICORR_BF16 ? 2 : 4;
  const int64_t H = w->d.hidden;
  size_t extra = align256(size_t(batch) * B * w->d.V * es);  // logits
  extra += align256(size_t(batch) * B * H * 2);               // slot_hidden
  extra += align256(size_t(batch) * H * 2);                   // target_state
  extra += align256(size_t(batch) * 4);                       // anchor ids
  extra += align256(size_t(batch) * B * 4);                   // tokens
  extra += align256(size_t(batch) * (B - 1) * 4);             // path score
  return base + extra;
}

lilicorr_status lilicorr_rerank_host(const lilicorr_weights* w, const void* logits_host,
                                     lilicorr_dtype ldtype, int64_t batch, int32_t B,
                                     int64_t V, int32_t K, const void* slot_hidden_host,
                                     const void* target_state_host,
                                     const int32_t* anchor_ids_host, int32_t* tokens_host,
                                     float* path_score_host, void* workspace,
                                     size_t workspace_bytes, void* stream_) {
  lilicorr_status st = check_call(w, ldtype, batch, B, V, K);
  if (st != LILICORR_OK) return st;
  if (!logits_host || !tokens_host || !path_score_host) return LILICORR_ERR_INVALID_ARG;
  const size_t need = lilicorr_workspace_bytes_host(w, batch, B, K, ldtype);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return LILICORR_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int es = ldtype == LILICORR_BF16 ? 2 : 4;
  const int64_t H = w->d.hidden;
  uint8_t* p = static_cast<uint8_t*>(workspace);
  const size_t base = lilicorr_workspace_bytes(w, batch, B, K);
  uint8_t* d_logits = p + base;
  uint8_t* d_hidden = d_logits + align256(size_t(batch) * B * V * es);
  uint8_t* d_target = d_hidden + align256(size_t(batch) * B * H * 2);
  uint8_t* d_anchor = d_target + align256(size_t(batch) * H * 2);
  uint8_t* d_tokens = d_anchor + align256(size_t(batch) * 4);
  uint8_t* d_path = d_tokens + align256(size_t(batch) * B * 4);
  if (slot_hidden_host)
    LC_CUDA(cudaMemcpyAsync(d_hidden, slot_hidden_host, size_t(batch) * B * H * 2,
                            cudaMemcpyHostToDevice, stream), "copy slot_hidden");
  if (target_state_host)
    LC_CUDA(cudaMemcpyAsync(d_target, target_state_host, size_t(batch) * H * 2,
                            cudaMemcpyHostToDevice, stream), "copy target_state");
  if (anchor_ids_host)
    LC_CUDA(cudaMemcpyAsync(d_anchor, anchor_ids_host, size_t(batch) * 4, cudaMemcpyHostToDevice,
                            stream), "copy anchor ids");
  // The logits arrive in chunks of blocks on a copy stream, rows 1..B-1 only (row 0, the
  // anchor position, is never read); each chunk's rerank starts on `stream` as soon as
  // its rows have landed, so the compute of one chunk hides under the copy of the next.
  // Chunks of at least K1_SPLIT_BELOW_ROWS rows (or one chunk): the logit pass splits rows
  // into segments only in calls of fewer rows, so every chunk then processes its rows
  // exactly as one call over the whole batch does, and the results are the same bits.
  const int64_t rows_all = batch * (B - 1);
  int64_t nchunk = std::min<int64_t>(std::min<int64_t>(batch, 8),
                                     std::max<int64_t>(1, rows_all / K1_SPLIT_BELOW_ROWS));
  int64_t per = (batch + nchunk - 1) / nchunk;
  while (nchunk > 1 && (batch - (nchunk - 1) * per) * (B - 1) < K1_SPLIT_BELOW_ROWS) {
    --nchunk;
    per = (batch + nchunk - 1) / nchunk;
  }
  cudaStream_t copy = nullptr;
  std::vector<cudaEvent_t> ev(size_t(nchunk) + 1, nullptr);
  auto cleanup = [&]() {
    for (auto& e : ev)
      if (e) cudaEventDestroy(e);
    if (copy) cudaStreamDestroy(copy);
  };
  cudaError_t ce = cudaStreamCreateWithFlags(&copy, cudaStreamNonBlocking);
  for (auto& e : ev)
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
  if (ce == cudaSuccess) ce = cudaEventRecord(ev[nchunk], stream);  // earlier work first
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(copy, ev[nchunk], 0);
  const size_t row = size_t(V) * es;
  for (int64_t c = 0; c < nchunk && ce == cudaSuccess; ++c) {
    const int64_t b0 = c * per, nb = std::min<int64_t>(per, batch - b0);
    if (nb <= 0) break;
    const size_t off = (size_t(b0) * B + 1) * row;
    ce = cudaMemcpy2DAsync(d_logits + off, size_t(B) * row,
                           static_cast<const uint8_t*>(logits_host) + off, size_t(B) * row,
                           size_t(B - 1) * row, size_t(nb), cudaMemcpyHostToDevice, copy);
    if (ce == cudaSuccess) ce = cudaEventRecord(ev[c], copy);
  }
  if (ce != cudaSuccess) {
    cleanup();
    return cuda_fail(ce, "copy logits");
  }
  for (int64_t c = 0; c < nchunk; ++c) {
    const int64_t b0 = c * per, nb = std::min<int64_t>(per, batch - b0);
    if (nb <= 0) break;
    ce = cudaStreamWaitEvent(stream, ev[c], 0);
    if (ce != cudaSuccess) {
      cleanup();
      return cuda_fail(ce, "cudaStreamWaitEvent");
    }
    st = lilicorr_rerank(
        w, d_logits + size_t(b0) * B * row, ldtype, nb, B, V, K,
        slot_hidden_host ? d_hidden + size_t(b0) * B * H * 2 : nullptr,
        target_state_host ? d_target + size_t(b0) * H * 2 : nullptr,
        anchor_ids_host ? reinterpret_cast<int32_t*>(d_anchor) + b0 : nullptr,
        reinterpret_cast<int32_t*>(d_tokens) + b0 * B, reinterpret_cast<float*>(d_path) + b0 * (B - 1),
        nullptr, p, base, stream_);
    if (st != LILICORR_OK) {
      cudaStreamSynchronize(stream);
      cleanup();
      return st;
    }
  }
  ce = cudaMemcpyAsync(tokens_host, d_tokens, size_t(batch) * B * 4, cudaMemcpyDeviceToHost,
                       stream);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(path_score_host, d_path, size_t(batch) * (B - 1) * 4,
                         cudaMemcpyDeviceToHost, stream);
  if (ce != cudaSuccess) {
    cudaStreamSynchronize(stream);
    cleanup();
    return cuda_fail(ce, "copy outputs");
  }
  ce = cudaStreamSynchronize(stream);
  cleanup();
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamSynchronize");
  return LILICORR_OK;
}

void lilicorr_stage_timing(int enable) {
  std::lock_guard<std::mutex> lk(g_timer.mu);
  g_timer.enabled = enable != 0;
}

int32_t lilicorr_stage_times(double* ms, int64_t* launches, int32_t n, int64_t* calls) {
  std::lock_guard<std::mutex> lk(g_timer.mu);
  for (auto& rec : g_timer.pending) {
    if (!rec.marks.empty()) cudaEventSynchronize(rec.marks.back().second);
    cudaEvent_t prev = rec.start;
    for (auto& m : rec.marks) {
      float t = 0.f;
      cudaEventElapsedTime(&t, prev, m.second);
      g_timer.ms[m.first] += t;
      g_timer.launches[m.first] += 1;
      prev = m.second;
    }
    cudaEventDestroy(rec.start);
    for (auto& m : rec.marks) cudaEventDestroy(m.second);
    g_timer.calls += 1;
  }
  g_timer.pending.clear();
  for (int s = 0; s < n && s < NSLOT; ++s) {
    if (ms) ms[s] = g_timer.ms[s];
    if (launches) launches[s] = g_timer.launches[s];
  }
  if (calls) *calls = g_timer.calls;
  for (int s = 0; s < NSLOT; ++s) {
    g_timer.ms[s] = 0;
    g_timer.launches[s] = 0;
  }
  g_timer.calls = 0;
  return NSLOT;
}

const char* lilicorr_stage_name(int32_t i) { return (i >= 0 && i < NSLOT) ? kSlotNames[i] : ""; }

}  // extern "C"
