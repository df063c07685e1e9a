// C ABI of libws: context, workspace layout and the host-side orchestration
// of the decoding path (include/ws.h documents every entry point).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <algorithm>
#include <vector>

#include "ws_flow.cuh"
#include "ws_internal.cuh"

// A weight matrix [rows, cols] (row-major, model dtype) and, for the tcgen05
// engine, its TMA tensor map (128-row boxes).
struct Mat {
  const void* p = nullptr;
  int rows = 0, cols = 0;
  TcMap map;
};

struct LayerW {
  Mat w_qkv, w_o, w_qc, w_kvc, w_oc, w_fc1, w_fc2;
  Mat w_kvrows;                 // rows k|v of w_qkv (drafter history projections)
  const void *b_q, *b_v, *b_o, *b_qc, *b_vc, *b_oc, *b_fc1, *b_fc2;
  const void *ln1_g, *ln1_b, *ln2_g, *ln2_b, *ln3_g, *ln3_b;
};

struct ws_ctx {
  ws_model_desc d;
  int es = 4;                   // element size of the model dtype
  int heads = 0, ppr = 0, n_pages = 0, n_xl = 0, max_split = 0;
  char* ws = nullptr;
  size_t ws_bytes = 0;
  const void *tok_emb = nullptr, *pos_emb = nullptr, *lnf_g = nullptr, *lnf_b = nullptr;
  Mat head, fuse_w;              // tied LM head (= tok_emb), fusion projection
  const void *lnh_g = nullptr, *lnh_b = nullptr, *mask_emb = nullptr;
  const void *dlnf_g = nullptr, *dlnf_b = nullptr;
  std::vector<LayerW> tl, dl;
  char* kv = nullptr;  size_t kv_layer_bytes = 0;     // target self KV pool
  char* hkv = nullptr;                                // drafter history KV pool
  void* xkv = nullptr; size_t x_slot_elems = 0, x_layer_elems = 0;
  int32_t* ptab = nullptr;
  float* rope = nullptr;
  int32_t *L = nullptr, *Fc = nullptr, *Fv = nullptr, *pend_start = nullptr, *pend_n = nullptr, *status = nullptr;
  int32_t* xcenter = nullptr;   // per slot: centre frame of the drafter's cross-attention window (-1: none)
  // verification-attention readout (ws_set_readout)
  int readout_layer = -1, half_width = 0, read_H = 0;
  void* qread = nullptr;        // the readout layer's cross-attention queries of the last verify [rows, d]
  float* rsc = nullptr;         // readout scores [max_batch][heads][max_frames]
  float2* rst = nullptr;        // readout softmax statistics [max_batch][heads]
  // candidate tree (ws_set_tree): row topology, drafter ranks, acceptance records
  int tree_n = 0;
  TreeMask tree = linear_tree();
  unsigned long long tree_parent4 = 0, tree_rank4 = 0;
  int32_t* tpath = nullptr;     // [max_batch][WS_TREE_REC]
  float* x = nullptr;
  void *h = nullptr, *q = nullptr, *ao = nullptr, *ffn = nullptr, *kb = nullptr, *vb = nullptr;
  float* hist = nullptr;
  unsigned long long* amax = nullptr;
  float* part = nullptr;
  void* feat = nullptr; float* hpre = nullptr; void* hh = nullptr;
  int pending_H = 0;
  unsigned long long cap_start = 0;   // launch counter when a capture began
  int max_fc = 0;
  const uint32_t* suppress = nullptr;
  int engine = WS_GEMM_SIMT;
  bool split_ok = false;        // split-K allowed (small-batch contexts)
  int mrows = 0;                // rows of the activation buffers
  AttnScratch as{};
  struct XMap { const void* base; TcMap bn[5]; };   // activation maps per token-tile width
  TcMap xkv_map, kv_map;        // acoustic K/V and target self K/V as [rows, 64] (tensor-core attention)
  std::vector<XMap> xmaps;
  bool pdl = true;              // programmatic dependent launch allowed
  bool cur_pdl = false;         // PDL for the call in progress (never on the legacy stream)
  // dataflow block verification (one-request bf16 contexts on the tcgen05 engine)
  bool flow_ok = false;         // eligible shape, set up and runnable on this device
  bool ln_in_gemm = true;       // layer norm inside eligible GEMMs (ws_fused_layernorm)
  bool flow_on = false;         // caller's switch (ws_fused_verify)
  int flow_grid = 0;
  const TcMap* fmaps = nullptr; // device: weight maps (16-row boxes), then head, ao, ffn, kv, xkv
  const FlowLayer* flayers = nullptr;
  int* fctr = nullptr;
  float* xpart = nullptr;
  float* f2part = nullptr;
  int max_groups = 0;           // cross-attention chunk groups per head
  int xs_rows = 0;              // residual rows per layer-norm staging pass
  float* conf = nullptr;        // drafted-token confidences [max_batch][K]
  float2* pstat = nullptr;      // acceptance scratch: (max, sum exp) per p / q logits row
  float2* qstat = nullptr;
  std::string err;
};

static std::atomic<unsigned long long> g_launches{0};

struct ws_graph {
  cudaGraphExec_t exec;
  unsigned long long kernels;   // kernel launches recorded in the graph
};
void ws_count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {

thread_local std::string g_err;

}  // namespace

void ws_set_thread_error(const char* msg) { g_err = msg ? msg : ""; }

namespace {

int fail(ws_ctx* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf; else g_err = buf;
  return code;
}

#define CK(x)                                                                                   \
  do {                                                                                          \
    cudaError_t e_ = (x);                                                                       \
    if (e_ != cudaSuccess) return fail(c, WS_ECUDA, "%s: %s", #x, cudaGetErrorString(e_));      \
  } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Element counts of the blobs (see ws.h).
size_t layer_elems(const ws_model_desc& d) {
  size_t D = d.d_model, F = d.d_ff;
  return 3 * D * D + D * D + D * D + 2 * D * D + D * D + F * D + D * F + 6 * D + F + D + 6 * D;
}
size_t target_elems(const ws_model_desc& d) {
  return (size_t)d.vocab * d.d_model + (size_t)d.max_pos * d.d_model + d.n_layers * layer_elems(d) + 2 * d.d_model;
}
size_t drafter_elems(const ws_model_desc& d) {
  if (d.drafter_layers == 0) return 0;
  size_t D = d.d_model;
  return D * (d.n_hist * D) + 5 * D + d.drafter_layers * layer_elems(d);
}

// Workspace layout: a bump allocator over the caller's buffer.
struct Layout {
  size_t off = 0;
  size_t take(size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; }
};

struct Plan {
  size_t tblob, dblob, kv, hkv, xkv, ptab, rope, state, x, h, q, ao, ffn, kb, vb, hist, amax, part, feat, hpre, hh;
  size_t acnt;
  size_t fmaps, flayers, fctr, xpart, f2part, pstat, qstat, conf, qread, rsc, rst, tpath;
  bool flow_shape;
  size_t kv_layer_bytes, total;
  int heads, ppr, n_pages, n_xl, max_split;
};

const char* check_desc(const ws_model_desc* d) {
  if (!d) return "null model description";
  if (d->dtype != WS_F32 && d->dtype != WS_BF16) return "dtype must be WS_F32 or WS_BF16";
  if (d->n_layers < 1 || d->n_layers > 256) return "n_layers out of range";
  if (d->d_model < 128 || d->d_model % 128 != 0 || d->d_model > 2048) return "d_model must be a multiple of 128, <= 2048";
  if (d->n_heads < 1 || d->d_model / d->n_heads != WS_DH || d->d_model % d->n_heads) return "d_model / n_heads must be 64";
  if (d->d_ff < 128 || d->d_ff % 128 != 0) return "d_ff must be a multiple of 128";
  if (d->vocab < 2 || d->vocab % 2 != 0 || d->vocab > 65536) return "vocab must be even, 2..65536";
  if (d->max_pos < 1 || d->max_pos > 4096) return "max_pos out of range";
  if (d->drafter_layers < 0 || d->drafter_layers > 8) return "drafter_layers out of range";
  if (d->K < 1 || d->K > 15) return "K must be 1..15";
  if (d->max_block < d->K + 1 || d->max_block > 16) return "max_block must be in K+1..16";
  if ((double)d->max_batch * ((d->max_pos + WS_PAGE - 1) / WS_PAGE) * 2 * d->n_heads * WS_PAGE * WS_DH >= 2147483648.0)
    return "self K/V pool of one layer must hold fewer than 2^31 elements";
  if (d->max_batch < 1 || d->max_batch > 4096) return "max_batch out of range";
  if (d->max_frames < 1 || d->max_frames > 4096) return "max_frames out of range";
  if (d->eos_id < 0 || d->eos_id >= d->vocab) return "eos_id outside the vocabulary";
  if (d->gemm < WS_GEMM_AUTO || d->gemm > WS_GEMM_TC) return "unknown gemm engine";
  if (d->drafter_layers > 0) {
    if (d->n_hist < 1 || d->n_hist > 8) return "n_hist must be 1..8";
    for (int i = 0; i < d->n_hist; ++i)
      if (d->hist_layers[i] < 0 || d->hist_layers[i] >= d->n_layers) return "history layer out of range";
  }
  return nullptr;
}

// Shapes the dataflow verify kernel handles: one request of <= 16 block rows,
// bf16, d a multiple of 256 up to 1280 (a compute warp's weight quarter of a
// 16-row task fits one 10 KB ring slot), the FFN a multiple of d, a decoder
// context of <= 576 positions (self-attention partials of <= 9 chunks).
bool flow_shape_ok(const ws_model_desc& d) {
  return d.dtype == WS_BF16 && d.max_batch == 1 && d.max_block <= FLOW_MAX_ROWS && d.d_model % 256 == 0 &&
         d.d_model <= 1280 && d.d_ff % d.d_model == 0 && d.d_ff / d.d_model <= 8 && d.n_heads <= 64 &&
         d.max_pos <= 576;
}

Plan make_plan(const ws_model_desc& d) {
  Plan p;
  Layout lay;
  const size_t es = d.dtype == WS_BF16 ? 2 : 4;
  const size_t D = d.d_model;
  p.heads = d.n_heads;
  p.ppr = (d.max_pos + WS_PAGE - 1) / WS_PAGE;
  p.n_pages = d.max_batch * p.ppr;
  p.n_xl = d.n_layers + d.drafter_layers;
  // attention splits: acoustic frames, cache positions, history positions + the drafter block
  p.max_split = std::max((d.max_frames + WS_XCHUNK - 1) / WS_XCHUNK, (d.max_pos + WS_XCHUNK - 1) / WS_XCHUNK + 1);
  const size_t M = (size_t)d.max_batch * d.max_block;
  p.tblob = lay.take(target_elems(d) * es);
  p.dblob = lay.take(drafter_elems(d) * es);
  p.kv_layer_bytes = (size_t)p.n_pages * 2 * d.n_heads * WS_PAGE * WS_DH * es;
  p.kv = lay.take(p.kv_layer_bytes * d.n_layers);
  p.hkv = lay.take(p.kv_layer_bytes * d.drafter_layers);
  p.xkv = lay.take((size_t)d.max_batch * p.n_xl * 2 * D * d.max_frames * es);
  p.ptab = lay.take((size_t)p.n_pages * 4);
  p.rope = lay.take((size_t)d.max_pos * WS_DH * 4);
  p.state = lay.take((size_t)d.max_batch * 6 * 4 + 256);
  p.x = lay.take(M * D * 4);
  p.h = lay.take(M * D * es);
  p.q = lay.take(M * D * es);
  p.ao = lay.take(M * D * es);
  p.ffn = lay.take(M * d.d_ff * es);
  p.kb = lay.take(M * D * es);
  p.vb = lay.take(M * D * es);
  const int nh = d.drafter_layers > 0 ? d.n_hist : 0;
  p.hist = lay.take((size_t)d.max_batch * d.max_block * nh * D * 4);
  p.amax = lay.take(M * 8);
  p.part = lay.take(M * d.n_heads * p.max_split * (WS_DH + 2) * 4);
  p.acnt = lay.take((size_t)d.max_batch * d.n_heads * 4);
  p.feat = lay.take(M * nh * D * es);
  p.hpre = lay.take(M * D * 4);
  p.hh = lay.take(M * D * es);
  // dataflow verify (one-request contexts): weight maps, layer table, counters, partials
  p.flow_shape = flow_shape_ok(d);
  const size_t fl = p.flow_shape ? 1 : 0;
  const size_t xgroups = ((d.max_frames + WS_XCHUNK - 1) / WS_XCHUNK + 3) / 4;
  p.fmaps = lay.take(fl * (6 * (size_t)d.n_layers + 6) * sizeof(TcMap));
  p.flayers = lay.take(fl * d.n_layers * sizeof(FlowLayer));
  p.fctr = lay.take(fl * ((size_t)d.n_layers * FLOW_CTR_LAYER + FLOW_CTR_GLOBAL) * 4);
  p.xpart = lay.take(fl * d.n_heads * xgroups * FLOW_MAX_ROWS * FLOW_GP * 4);
  p.f2part = lay.take(fl * (D / 16) * (d.d_ff / std::max(1, d.d_model)) * 256 * 4);
  p.conf = lay.take((size_t)d.max_batch * d.K * 4);   // drafted-token confidences
  p.qread = lay.take(M * D * es);                      // readout: queries of the readout layer
  p.rsc = lay.take((size_t)d.max_batch * d.n_heads * d.max_frames * 4);
  p.rst = lay.take((size_t)d.max_batch * d.n_heads * 8);
  p.tpath = lay.take((size_t)d.max_batch * WS_TREE_REC * 4);   // tree acceptance records
  p.pstat = lay.take(M * 8);        // sampling acceptance: softmax statistics per logits row
  p.qstat = lay.take(M * 8);
  p.total = lay.off;
  return p;
}

void bind_layer(LayerW& w, const char*& p, const ws_model_desc& d, size_t es) {
  const size_t D = d.d_model, F = d.d_ff;
  auto take = [&](size_t n) { const void* r = p; p += n * es; return r; };
  auto mat = [&](Mat& m, size_t rows, size_t cols) { m.p = take(rows * cols); m.rows = (int)rows; m.cols = (int)cols; };
  mat(w.w_qkv, 3 * D, D); mat(w.w_o, D, D); mat(w.w_qc, D, D); mat(w.w_kvc, 2 * D, D);
  mat(w.w_oc, D, D); mat(w.w_fc1, F, D); mat(w.w_fc2, D, F);
  w.w_kvrows.p = (const char*)w.w_qkv.p + D * D * es; w.w_kvrows.rows = (int)(2 * D); w.w_kvrows.cols = (int)D;
  w.b_q = take(D); w.b_v = take(D); w.b_o = take(D); w.b_qc = take(D); w.b_vc = take(D); w.b_oc = take(D);
  w.b_fc1 = take(F); w.b_fc2 = take(D);
  w.ln1_g = take(D); w.ln1_b = take(D); w.ln2_g = take(D); w.ln2_b = take(D); w.ln3_g = take(D); w.ln3_b = take(D);
}

KVPool pool(ws_ctx* c, char* base, int layer) {
  KVPool k;
  k.base = base + (size_t)layer * c->kv_layer_bytes;
  k.ptab = c->ptab;
  k.ppr = c->ppr;
  k.n_heads = c->heads;
  return k;
}

XKV xkv_of(ws_ctx* c) {
  XKV x;
  x.base = c->xkv;
  x.slot_stride = c->x_slot_elems;
  x.layer_stride = c->x_layer_elems;
  x.max_frames = c->d.max_frames;
  x.n_heads = c->heads;
  return x;
}

Epi epi0(ws_ctx* c, int kind) {
  Epi e;
  memset(&e, 0, sizeof e);
  e.kind = kind;
  e.d = c->d.d_model;
  e.status = c->status;
  e.rope = c->rope;
  e.suppress = c->suppress;
  e.max_block = c->d.max_block;
  return e;
}

// Split-K factor of a weight shape: a function of (N, K) and the context only,
// never of the token count, so every row is reduced in the same order.
// Only small-batch contexts split: their tiles are at most 64 tokens wide, so
// the fp32 partials folded through distributed shared memory stay small.
int splits_for(const ws_ctx* c, int N, int K) {
  if (!c->split_ok) return 1;
  const int tiles = (N + 127) / 128, kb = K / 64;
  if (tiles >= 100) return 1;
  int s = (148 + tiles - 1) / tiles;
  s = std::min(s, std::max(1, kb / 2));
  return std::max(1, std::min(s, 8));       // one portable thread-block cluster per tile
}

// Y = X W^T with a fused epilogue.  X has x_rows allocated rows.
struct LnIn {
  const float* x;
  const void* g;
  const void* b;
};

template <typename T>
cudaError_t gemm(ws_ctx* c, const void* X, uint64_t x_rows, const Mat& W, int M, const Epi& e, cudaStream_t s,
                 int batch = 1, bool allow_split = true, const LnIn* ln = nullptr) {
  GemmShape g;
  g.X = X; g.ldx = W.cols; g.W = W.p; g.ldw = W.cols; g.M = M; g.N = W.rows; g.K = W.cols; g.batch = batch;
  if (ln) { g.ln_x = ln->x; g.ln_g = ln->g; g.ln_b = ln->b; }
  if (c->engine == WS_GEMM_TC && sizeof(T) == 2)
  {
    const TcMap* mx = nullptr;
    for (const auto& xm : c->xmaps)
      if (xm.base == X) { mx = &xm.bn[tc_bn_index(tc_pick_bn(M, g.N, batch))]; break; }
    return launch_gemm_tc(g, e, W.map, mx, X, x_rows, allow_split ? splits_for(c, g.N, g.K) : 1, s,
                          c->cur_pdl);
  }
  return launch_gemm_simt<T>(g, e, s, c->cur_pdl);
}

template <typename T>
cudaError_t layernorm(ws_ctx* c, int M, const float* x, const void* g, const void* b, void* y,
                      cudaStream_t s, int group_skip = 0);

// Y = LayerNorm(x) W^T.  Small split-K calls on the tcgen05 engine normalise
// inside the GEMM (bit-identical operand); otherwise a layer-norm kernel
// writes c->h and the GEMM reads it.
template <typename T>
cudaError_t ln_gemm(ws_ctx* c, int M, const float* x, const void* g, const void* b, const Mat& W, const Epi& e,
                    cudaStream_t s, int group_skip = 0) {
  if (sizeof(T) == 2 && group_skip == 0 && c->ln_in_gemm && c->engine == WS_GEMM_TC &&
      tc_ln_input_ok(M, W.rows, W.cols, splits_for(c, W.rows, W.cols))) {
    const LnIn ln = {x, g, b};
    return gemm<T>(c, c->h, c->mrows, W, M, e, s, 1, true, &ln);
  }
  cudaError_t r = layernorm<T>(c, M, x, g, b, c->h, s, group_skip);
  if (r != cudaSuccess) return r;
  return gemm<T>(c, c->h, c->mrows, W, M, e, s);
}

template <typename T>
cudaError_t layernorm(ws_ctx* c, int M, const float* x, const void* g, const void* b, void* y,
                      cudaStream_t s, int group_skip) {
  const int D = c->d.d_model;
  return launch_layernorm<T>(M, D, x, D, (const T*)g, (const T*)b, (T*)y, D, group_skip, s, c->cur_pdl);
}

bool is_hist_layer(const ws_model_desc& d, int l, int& idx) {
  if (d.drafter_layers == 0) return false;
  for (int i = 0; i < d.n_hist; ++i)
    if (d.hist_layers[i] == l) { idx = i; return true; }
  return false;
}

// --------------------------------------------------------------------------- dataflow verify
// Weight maps with 16-row boxes for every projection and the LM head, the
// activation / K/V maps the kernel loads with, and the per-layer table, all
// copied to the device once.  Leaves flow_ok false when the shape or the
// device does not allow the kernel.
cudaError_t setup_flow(ws_ctx* c, const Plan& p, cudaStream_t s) {
  const ws_model_desc& d = c->d;
  if (!p.flow_shape || c->engine != WS_GEMM_TC || !c->as.kv_map || !c->as.xkv_map) return cudaSuccess;
  const int grid = flow_prepare();
  cudaGetLastError();                 // a device that cannot run it is not an error
  if (grid <= 0) return cudaSuccess;
  std::vector<TcMap> maps;
  bool ok = true;
  auto map16 = [&](const Mat& m) {
    TcMap t;
    ok = ok && tc_encode_map(&t, m.p, (uint64_t)m.rows, (uint64_t)m.cols, 16);
    maps.push_back(t);
  };
  for (const LayerW& w : c->tl) {
    map16(w.w_qkv); map16(w.w_o); map16(w.w_qc); map16(w.w_oc); map16(w.w_fc1); map16(w.w_fc2);
  }
  map16(c->head);
  const TcMap* ao = nullptr;
  const TcMap* ffn = nullptr;
  for (const auto& xm : c->xmaps) {
    if (xm.base == c->ao) ao = &xm.bn[0];
    if (xm.base == c->ffn) ffn = &xm.bn[0];
  }
  if (!ok || !ao || !ffn) return cudaSuccess;
  maps.push_back(*ao); maps.push_back(*ffn); maps.push_back(c->kv_map); maps.push_back(c->xkv_map);
  // residual rows for the layer norms: whole fp32 rows, as many as the staging buffer holds
  const int xs_rows = std::min(FLOW_MAX_ROWS, FLOW_XS_BYTES / (4 * d.d_model));
  TcMap xm;
  if (!tc_encode_rows_f32(&xm, c->x, (uint64_t)c->mrows, (uint64_t)d.d_model, (uint32_t)xs_rows))
    return cudaSuccess;
  maps.push_back(xm);
  TcMap* dm = (TcMap*)(c->ws + p.fmaps);
  std::vector<FlowLayer> fl(d.n_layers);
  for (int l = 0; l < d.n_layers; ++l) {
    const LayerW& w = c->tl[l];
    FlowLayer& f = fl[l];
    f.map_qkv = dm + 6 * l; f.map_o = dm + 6 * l + 1; f.map_qc = dm + 6 * l + 2;
    f.map_oc = dm + 6 * l + 3; f.map_fc1 = dm + 6 * l + 4; f.map_fc2 = dm + 6 * l + 5;
    f.b_q = (const bf16*)w.b_q; f.b_v = (const bf16*)w.b_v; f.b_o = (const bf16*)w.b_o;
    f.b_qc = (const bf16*)w.b_qc; f.b_oc = (const bf16*)w.b_oc; f.b_fc1 = (const bf16*)w.b_fc1;
    f.b_fc2 = (const bf16*)w.b_fc2;
    f.ln1_g = (const bf16*)w.ln1_g; f.ln1_b = (const bf16*)w.ln1_b; f.ln2_g = (const bf16*)w.ln2_g;
    f.ln2_b = (const bf16*)w.ln2_b; f.ln3_g = (const bf16*)w.ln3_g; f.ln3_b = (const bf16*)w.ln3_b;
    int hidx = -1;
    f.hist_idx = is_hist_layer(d, l, hidx) ? hidx : -1;
  }
  cudaError_t e = cudaMemcpyAsync(dm, maps.data(), maps.size() * sizeof(TcMap), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->ws + p.flayers, fl.data(), fl.size() * sizeof(FlowLayer), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(c->ws + p.fctr, 0, ((size_t)d.n_layers * FLOW_CTR_LAYER + FLOW_CTR_GLOBAL) * 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);    // host vectors go out of scope
  if (e != cudaSuccess) return e;
  c->fmaps = dm;
  c->flayers = (const FlowLayer*)(c->ws + p.flayers);
  c->fctr = (int*)(c->ws + p.fctr);
  c->xpart = (float*)(c->ws + p.xpart);
  c->f2part = (float*)(c->ws + p.f2part);
  c->max_groups = ((d.max_frames + WS_XCHUNK - 1) / WS_XCHUNK + 3) / 4;
  c->xs_rows = xs_rows;
  c->flow_grid = grid;
  c->flow_ok = true;
  return cudaSuccess;
}

int flow_verify(ws_ctx* c, const int32_t* req, int H, const int32_t* block, const int32_t* blen, int32_t* target,
                float* logits, cudaStream_t s) {
  const ws_model_desc& d = c->d;
  const int nL = d.n_layers;
  FlowArgs a;
  memset(&a, 0, sizeof a);
  a.layers = c->flayers;
  a.map_head = c->fmaps + 6 * nL; a.map_ao = c->fmaps + 6 * nL + 1; a.map_ffn = c->fmaps + 6 * nL + 2;
  a.map_kv = c->fmaps + 6 * nL + 3; a.map_xkv = c->fmaps + 6 * nL + 4; a.map_x = c->fmaps + 6 * nL + 5;
  a.xs_rows = c->xs_rows;
  a.n_layers = nL; a.d = d.d_model; a.f = d.d_ff; a.heads = c->heads; a.V = d.vocab; a.max_pos = d.max_pos;
  a.max_block = d.max_block; a.n_hist = d.drafter_layers > 0 ? d.n_hist : 0;
  a.H = H; a.req_ids = req; a.block = block; a.block_len = blen;
  a.tok_emb = (const bf16*)c->tok_emb; a.pos_emb = (const bf16*)c->pos_emb;
  a.lnf_g = (const bf16*)c->lnf_g; a.lnf_b = (const bf16*)c->lnf_b;
  a.x = c->x; a.q = (bf16*)c->q; a.ao = (bf16*)c->ao; a.ffn = (bf16*)c->ffn;
  a.L = c->L; a.Fv = c->Fv; a.pend_start = c->pend_start; a.pend_n = c->pend_n;
  a.kv = c->kv; a.kv_layer_bytes = c->kv_layer_bytes; a.ptab = c->ptab; a.ppr = c->ppr;
  a.xkv_slot_rows = c->x_slot_elems / WS_DH; a.xkv_layer_rows = c->x_layer_elems / WS_DH;
  a.max_frames = d.max_frames;
  a.hist = c->hist; a.xpart = c->xpart; a.max_groups = c->max_groups; a.fpart = c->f2part;
  a.amax = c->amax; a.logits = logits; a.suppress = c->suppress; a.target = target;
  a.ctr = c->fctr; a.status = c->status;
  CK(launch_flow_verify(a, c->flow_grid, s));
  if (d.drafter_layers > 0) c->pending_H = H > c->pending_H ? H : c->pending_H;
  return WS_OK;
}

// --------------------------------------------------------------------------- verify
template <typename T>
int verify_impl(ws_ctx* c, int n, const int32_t* req, int H, const int32_t* block, const int32_t* blen,
                int32_t* target, float* logits, cudaStream_t s, const TreeMask* tree = nullptr) {
  const ws_model_desc& d = c->d;
  const int D = d.d_model, M = n * H;
  if (sizeof(T) == 2 && c->flow_ok && c->flow_on && c->readout_layer < 0 && !tree && n == 1 && H <= FLOW_MAX_ROWS)
    return flow_verify(c, req, H, block, blen, target, logits, s);
  const TreeMask tm = tree ? *tree : linear_tree();
  c->read_H = H;
  const bool pdl = c->cur_pdl;
  RowMap rm;
  rm.mode = ROW_VERIFY; rm.H = H; rm.max_pos = d.max_pos; rm.req_ids = req; rm.L = c->L;
  rm.block_len = blen; rm.pend_start = c->pend_start; rm.pend_n = c->pend_n;
  CK(launch_embed_target<T>(n, H, rm, tm.depth4, block, (const T*)c->tok_emb, (const T*)c->pos_emb, D, d.vocab,
                            c->x, c->pend_start, c->pend_n, c->status, s, pdl));
  for (int l = 0; l < d.n_layers; ++l) {
    const LayerW& w = c->tl[l];
    Epi e = epi0(c, EPI_QKV);
    e.bias = w.b_q; e.bias2 = w.b_v; e.out = c->q; e.rm = rm; e.kv = pool(c, c->kv, l);
    CK(ln_gemm<T>(c, M, c->x, w.ln1_g, w.ln1_b, w.w_qkv, e, s));
    CK(launch_self_attn<T>(n, H, rm, tm, (const T*)c->q, pool(c, c->kv, l), (T*)c->ao, c->heads, c->as, s, pdl));
    e = epi0(c, EPI_RESID);
    e.bias = w.b_o; e.resid = c->x; e.ldr = D;
    CK(gemm<T>(c, c->ao, c->mrows, w.w_o, M, e, s));
    e = epi0(c, EPI_STORE);
    e.bias = w.b_qc; e.out = c->q; e.ldo = D;
    CK(ln_gemm<T>(c, M, c->x, w.ln2_g, w.ln2_b, w.w_qc, e, s));
    if (l == c->readout_layer) CK(cudaMemcpyAsync(c->qread, c->q, (size_t)M * D * c->es, cudaMemcpyDeviceToDevice, s));
    CK(launch_cross_attn<T>(n, H, req, c->Fv, (const T*)c->q, xkv_of(c), l, (T*)c->ao, c->heads, c->max_fc, c->as,
                            s, pdl));
    e = epi0(c, EPI_RESID);
    e.bias = w.b_oc; e.resid = c->x; e.ldr = D;
    CK(gemm<T>(c, c->ao, c->mrows, w.w_oc, M, e, s));
    e = epi0(c, EPI_GELU);
    e.bias = w.b_fc1; e.out = c->ffn; e.ldo = d.d_ff;
    CK(ln_gemm<T>(c, M, c->x, w.ln3_g, w.ln3_b, w.w_fc1, e, s));
    e = epi0(c, EPI_RESID);
    e.bias = w.b_fc2; e.resid = c->x; e.ldr = D;
    int hidx;
    if (is_hist_layer(d, l, hidx)) {
      e.hist = c->hist; e.hist_idx = hidx; e.n_hist = d.n_hist; e.rm = rm;
    }
    CK(gemm<T>(c, c->ffn, c->mrows, w.w_fc2, M, e, s));
  }
  CK(launch_argmax_init(M, c->amax, s, pdl));
  Epi e = epi0(c, EPI_LOGITS);
  e.logits = logits; e.ldl = d.vocab; e.amax = c->amax;
  CK(ln_gemm<T>(c, M, c->x, c->lnf_g, c->lnf_b, c->head, e, s));
  CK(launch_argmax_finalize(n, H, blen, c->amax, target, H, 0, s, pdl));
  if (d.drafter_layers > 0) c->pending_H = H > c->pending_H ? H : c->pending_H;
  return WS_OK;
}

// --------------------------------------------------------------------------- draft
template <typename T>
int draft_impl(ws_ctx* c, int n, const int32_t* req, int32_t* block, float temp, uint64_t seed, uint64_t rnd,
               float* q_logits, cudaStream_t s) {
  const ws_model_desc& d = c->d;
  const int D = d.d_model, K = d.K, K1 = K + 1;
  const bool pdl = c->cur_pdl;
  // 1) fold the rows of the last verify into the drafter history
  const int Hp = c->pending_H;
  if (Hp > 0) {
    const int Mh = n * Hp;
    CK(launch_hist_gather<T>(n, Hp, req, c->pend_n, c->hist, d.max_block, d.n_hist, D, (T*)c->feat, s, pdl));
    Epi e = epi0(c, EPI_F32);
    e.out = c->hpre; e.ldo = D;
    CK(gemm<T>(c, c->feat, c->mrows, c->fuse_w, Mh, e, s));
    CK(layernorm<T>(c, Mh, c->hpre, c->lnh_g, c->lnh_b, c->hh, s));
    RowMap rh;
    rh.mode = ROW_HIST; rh.H = Hp; rh.max_pos = d.max_pos; rh.req_ids = req; rh.L = c->L;
    rh.block_len = nullptr; rh.pend_start = c->pend_start; rh.pend_n = c->pend_n;
    for (int l = 0; l < d.drafter_layers; ++l) {
      const LayerW& w = c->dl[l];
      Epi eh = epi0(c, EPI_HISTKV);
      eh.bias2 = w.b_v; eh.rm = rh; eh.kv = pool(c, c->hkv, l);
      CK(gemm<T>(c, c->hh, c->mrows, w.w_kvrows, Mh, eh, s));
    }
  }
  // 2) the block X_t = [Emb(anchor), m, ..., m] through the drafter layers
  const int M = n * K1;
  RowMap rd;
  rd.mode = ROW_DRAFT; rd.H = K1; rd.max_pos = d.max_pos; rd.req_ids = req; rd.L = c->L;
  rd.block_len = nullptr; rd.pend_start = c->pend_start; rd.pend_n = c->pend_n;
  CK(launch_embed_draft<T>(n, K1, req, block, (const T*)c->tok_emb, (const T*)c->mask_emb, D, d.vocab, c->x,
                           c->pend_n, c->status, s, pdl));
  for (int l = 0; l < d.drafter_layers; ++l) {
    const LayerW& w = c->dl[l];
    Epi e = epi0(c, EPI_QKV_DRAFT);
    e.bias = w.b_q; e.bias2 = w.b_v; e.out = c->q; e.kout = c->kb; e.vout = c->vb; e.rm = rd;
    CK(ln_gemm<T>(c, M, c->x, w.ln1_g, w.ln1_b, w.w_qkv, e, s));
    CK(launch_draft_attn<T>(n, K1, req, c->L, (const T*)c->q, (const T*)c->kb, (const T*)c->vb,
                            pool(c, c->hkv, l), (T*)c->ao, c->heads, d.max_pos, c->as, s, pdl));
    e = epi0(c, EPI_RESID);
    e.bias = w.b_o; e.resid = c->x; e.ldr = D;
    CK(gemm<T>(c, c->ao, c->mrows, w.w_o, M, e, s));
    e = epi0(c, EPI_STORE);
    e.bias = w.b_qc; e.out = c->q; e.ldo = D;
    CK(ln_gemm<T>(c, M, c->x, w.ln2_g, w.ln2_b, w.w_qc, e, s));
    if (c->half_width > 0)
      CK(launch_window_attn<T>(n, K1, req, c->Fv, c->xcenter, c->half_width, (const T*)c->q, D, xkv_of(c),
                               d.n_layers + l, (T*)c->ao, s, pdl));
    else
      CK(launch_cross_attn<T>(n, K1, req, c->Fv, (const T*)c->q, xkv_of(c), d.n_layers + l, (T*)c->ao, c->heads,
                              c->max_fc, c->as, s, pdl));
    e = epi0(c, EPI_RESID);
    e.bias = w.b_oc; e.resid = c->x; e.ldr = D;
    CK(gemm<T>(c, c->ao, c->mrows, w.w_oc, M, e, s));
    e = epi0(c, EPI_GELU);
    e.bias = w.b_fc1; e.out = c->ffn; e.ldo = d.d_ff;
    CK(ln_gemm<T>(c, M, c->x, w.ln3_g, w.ln3_b, w.w_fc1, e, s));
    e = epi0(c, EPI_RESID);
    e.bias = w.b_fc2; e.resid = c->x; e.ldr = D;
    CK(gemm<T>(c, c->ffn, c->mrows, w.w_fc2, M, e, s));
  }
  // 3) final LN on the K mask rows, shared LM head, argmax or sampling
  const int Mk = n * K;
  Epi e = epi0(c, EPI_LOGITS);
  e.logits = q_logits; e.ldl = d.vocab;
  if (temp <= 0.0f) {
    CK(launch_argmax_init(Mk, c->amax, s, pdl));
    e.amax = c->amax;
    CK(ln_gemm<T>(c, Mk, c->x, c->dlnf_g, c->dlnf_b, c->head, e, s, K1));
    CK(launch_argmax_finalize(n, K, nullptr, c->amax, block, K1, 1, s, pdl));
  } else {
    CK(ln_gemm<T>(c, Mk, c->x, c->dlnf_g, c->dlnf_b, c->head, e, s, K1));
    CK(launch_sample_rows(n, K, req, q_logits, d.vocab, d.vocab, temp, seed, rnd, c->suppress, block, K1, 1, s,
                          pdl));
  }
  return WS_OK;
}

// --------------------------------------------------------------------------- cross K/V
template <typename T>
int cross_kv_impl(ws_ctx* c, int n, const int32_t* req, const void* enc, const int32_t* cu, const int32_t* valid,
                  int maxF, int total_frames, cudaStream_t s) {
  const ws_model_desc& d = c->d;
  CK(launch_set_frames(n, req, cu, valid, d.max_frames, c->Fc, c->Fv, c->status, s));
  for (int l = 0; l < c->n_xl; ++l) {
    const LayerW& w = l < d.n_layers ? c->tl[l] : c->dl[l - d.n_layers];
    Epi e = epi0(c, EPI_CROSSKV);
    e.bias2 = w.b_vc; e.xkv = xkv_of(c); e.xlayer = l; e.cu_frames = cu; e.req_ids = req;
    CK(gemm<T>(c, enc, (uint64_t)total_frames, w.w_kvc, maxF, e, s, n, false));
  }
  if (maxF > c->max_fc) c->max_fc = maxF;
  return WS_OK;
}

int check_common(ws_ctx* c, int n, const int32_t* req, ws_stream stream = nullptr) {
  if (!c) return fail(nullptr, WS_EINVAL, "null context");
  // PDL only on created streams; the legacy default stream serialises plainly
  c->cur_pdl = c->pdl && stream != nullptr && (cudaStream_t)stream != cudaStreamLegacy &&
               (cudaStream_t)stream != cudaStreamPerThread;
  if (n < 0 || n > c->d.max_batch) return fail(c, WS_EINVAL, "n_req %d outside 0..max_batch (%d)", n, c->d.max_batch);
  if (n > 0 && !req) return fail(c, WS_EINVAL, "null req_ids");
  return WS_OK;
}

}  // namespace

// =========================================================================== C ABI
extern "C" {

size_t ws_query_workspace(const ws_model_desc* desc) {
  if (check_desc(desc)) return 0;
  return make_plan(*desc).total;
}

int ws_load_weights(ws_ctx** out, const ws_model_desc* desc, void* workspace, size_t workspace_bytes,
                    const void* target_blob, const void* drafter_blob, ws_stream stream) {
  ws_ctx* c = nullptr;
  if (!out) return fail(nullptr, WS_EINVAL, "null output handle");
  *out = nullptr;
  if (const char* why = check_desc(desc)) return fail(nullptr, WS_EINVAL, "%s", why);
  if (!workspace || ((uintptr_t)workspace & 255)) return fail(nullptr, WS_EINVAL, "workspace null or not 256-byte aligned");
  if (!target_blob) return fail(nullptr, WS_EINVAL, "null target blob");
  if (desc->drafter_layers > 0 && !drafter_blob) return fail(nullptr, WS_EINVAL, "null drafter blob");
  Plan p = make_plan(*desc);
  if (workspace_bytes < p.total)
    return fail(nullptr, WS_ENOSPACE, "workspace %zu bytes < required %zu", workspace_bytes, p.total);
  if (desc->gemm == WS_GEMM_TC && !tc_engine_available())
    return fail(nullptr, WS_EUNSUPPORTED, "tcgen05 GEMM engine not built");

  c = new ws_ctx();
  c->d = *desc;
  c->es = desc->dtype == WS_BF16 ? 2 : 4;
  c->heads = p.heads; c->ppr = p.ppr; c->n_pages = p.n_pages; c->n_xl = p.n_xl; c->max_split = p.max_split;
  c->ws = (char*)workspace; c->ws_bytes = workspace_bytes;
  c->engine = (desc->gemm == WS_GEMM_TC || (desc->gemm == WS_GEMM_AUTO && desc->dtype == WS_BF16 &&
                                            tc_engine_available())) ? WS_GEMM_TC : WS_GEMM_SIMT;
  char* b = c->ws;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t tb = target_elems(*desc) * c->es, db = drafter_elems(*desc) * c->es;
  auto cleanup = [&](int code) { delete c; return code; };
  cudaError_t e = cudaMemcpyAsync(b + p.tblob, target_blob, tb, cudaMemcpyDefault, s);
  if (e == cudaSuccess && db) e = cudaMemcpyAsync(b + p.dblob, drafter_blob, db, cudaMemcpyDefault, s);
  if (e != cudaSuccess) { fail(nullptr, WS_ECUDA, "weight copy: %s", cudaGetErrorString(e)); return cleanup(WS_ECUDA); }

  const char* tp = b + p.tblob;
  const size_t D = desc->d_model;
  c->tok_emb = tp; tp += (size_t)desc->vocab * D * c->es;
  c->head.p = c->tok_emb; c->head.rows = desc->vocab; c->head.cols = (int)D;
  c->pos_emb = tp; tp += (size_t)desc->max_pos * D * c->es;
  c->tl.resize(desc->n_layers);
  for (auto& w : c->tl) bind_layer(w, tp, *desc, c->es);
  c->lnf_g = tp; tp += D * c->es;
  c->lnf_b = tp;
  if (desc->drafter_layers > 0) {
    const char* dp = b + p.dblob;
    c->fuse_w.p = dp; c->fuse_w.rows = (int)D; c->fuse_w.cols = (int)(desc->n_hist * D);
    dp += D * desc->n_hist * D * c->es;
    c->lnh_g = dp; dp += D * c->es;
    c->lnh_b = dp; dp += D * c->es;
    c->mask_emb = dp; dp += D * c->es;
    c->dlnf_g = dp; dp += D * c->es;
    c->dlnf_b = dp; dp += D * c->es;
    c->dl.resize(desc->drafter_layers);
    for (auto& w : c->dl) bind_layer(w, dp, *desc, c->es);
  }
  c->kv = b + p.kv; c->kv_layer_bytes = p.kv_layer_bytes;
  c->hkv = b + p.hkv;
  c->xkv = b + p.xkv;
  c->x_layer_elems = 2 * D * desc->max_frames;
  c->x_slot_elems = c->x_layer_elems * p.n_xl;
  c->ptab = (int32_t*)(b + p.ptab);
  c->rope = (float*)(b + p.rope);
  int32_t* st = (int32_t*)(b + p.state);
  c->L = st; c->Fc = st + desc->max_batch; c->Fv = st + 2 * desc->max_batch;
  c->pend_start = st + 3 * desc->max_batch; c->pend_n = st + 4 * desc->max_batch;
  c->status = st + 5 * desc->max_batch;
  c->xcenter = st + 5 * desc->max_batch + 64;     // after the status word (its 256-byte pad)
  c->x = (float*)(b + p.x); c->h = b + p.h; c->q = b + p.q; c->ao = b + p.ao; c->ffn = b + p.ffn;
  c->kb = b + p.kb; c->vb = b + p.vb; c->hist = (float*)(b + p.hist);
  c->amax = (unsigned long long*)(b + p.amax); c->part = (float*)(b + p.part);
  c->as.part = c->part; c->as.counters = (int*)(b + p.acnt); c->as.status = st + 5 * desc->max_batch;
  c->feat = b + p.feat; c->hpre = (float*)(b + p.hpre); c->hh = b + p.hh;
  c->pstat = (float2*)(b + p.pstat); c->qstat = (float2*)(b + p.qstat); c->conf = (float*)(b + p.conf);
  c->qread = b + p.qread; c->rsc = (float*)(b + p.rsc); c->rst = (float2*)(b + p.rst);
  c->tpath = (int32_t*)(b + p.tpath);
  c->mrows = desc->max_batch * desc->max_block;
  c->split_ok = c->mrows <= 64;
  if (c->engine == WS_GEMM_TC) {
    bool ok = true;
    auto enc = [&](Mat& m) { ok = ok && tc_encode_map(&m.map, m.p, (uint64_t)m.rows, (uint64_t)m.cols, 128); };
    for (auto* L : {&c->tl, &c->dl})
      for (auto& w : *L) {
        enc(w.w_qkv); enc(w.w_o); enc(w.w_qc); enc(w.w_kvc); enc(w.w_oc); enc(w.w_fc1); enc(w.w_fc2);
        enc(w.w_kvrows);
      }
    enc(c->head);
    if (desc->drafter_layers > 0) enc(c->fuse_w);
    // activation buffers: one map per token-tile width
    auto xm = [&](const void* base, int cols) {
      ws_ctx::XMap m;
      m.base = base;
      const int bns[5] = {16, 32, 64, 128, 256};
      for (int i = 0; i < 5; ++i) ok = ok && tc_encode_map(&m.bn[i], base, (uint64_t)c->mrows, (uint64_t)cols, bns[i]);
      c->xmaps.push_back(m);
    };
    xm(c->h, (int)D); xm(c->ao, (int)D); xm(c->ffn, desc->d_ff); xm(c->hh, (int)D);
    // tensor-core attention: K/V chunks as 64 x 64 boxes of [rows, 64] matrices
    ok = ok && tc_encode_map(&c->xkv_map, c->xkv, (uint64_t)desc->max_batch * c->x_slot_elems / WS_DH, WS_DH, 64);
    ok = ok && tc_encode_map(&c->kv_map, c->kv, (uint64_t)desc->n_layers * p.kv_layer_bytes / (WS_DH * 2), WS_DH, 64);
    if (ok) { c->as.xkv_map = &c->xkv_map; c->as.kv_map = &c->kv_map; c->as.kv_base = c->kv; }
    if (desc->drafter_layers > 0) xm(c->feat, (int)(desc->n_hist * D));
    if (ok && tc_init_attributes() != cudaSuccess) ok = false;
    if (!ok) { fail(nullptr, WS_ECUDA, "TMA descriptor encoding failed"); return cleanup(WS_ECUDA); }
  }

  std::vector<int32_t> pt(p.n_pages);
  for (int i = 0; i < p.n_pages; ++i) pt[i] = i;   // each slot owns its own pages
  e = cudaMemcpyAsync(c->ptab, pt.data(), pt.size() * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(st, 0, (size_t)desc->max_batch * 5 * 4 + 256, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->xcenter, 0xFF, (size_t)desc->max_batch * 4, s);   // -1: no centre
  if (e == cudaSuccess) e = cudaMemsetAsync(c->hist, 0, (size_t)desc->max_batch * desc->max_block *
                                                        (desc->drafter_layers ? desc->n_hist : 0) * D * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->as.counters, 0, (size_t)desc->max_batch * desc->n_heads * 4, s);
  if (e == cudaSuccess) e = desc->dtype == WS_BF16 ? attn_init_attributes<bf16>() : attn_init_attributes<float>();
  if (e == cudaSuccess) e = launch_rope_table(c->rope, desc->max_pos, s);
  // caches start at zero: masked keys beyond a request's length or frames
  // then hold finite values (the probabilities of masked keys are exact zeros)
  if (e == cudaSuccess) e = cudaMemsetAsync(c->kv, 0, p.kv_layer_bytes * desc->n_layers, s);
  if (e == cudaSuccess && desc->drafter_layers > 0)
    e = cudaMemsetAsync(c->hkv, 0, p.kv_layer_bytes * desc->drafter_layers, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->xkv, 0, (size_t)desc->max_batch * c->x_slot_elems * c->es, s);
  if (e == cudaSuccess) e = setup_flow(c, p, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) { fail(nullptr, WS_ECUDA, "context init: %s", cudaGetErrorString(e)); return cleanup(WS_ECUDA); }
  *out = c;
  return WS_OK;
}

int ws_reset(ws_ctx* c, int n, const int32_t* req, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  CK(launch_reset(n, req, c->L, c->pend_n, c->xcenter, (cudaStream_t)stream));
  return WS_OK;
}

int ws_cross_kv(ws_ctx* c, int n, const int32_t* req, const void* enc, const int32_t* cu, const int32_t* valid,
                int maxF, int total_frames, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (!enc || !cu) return fail(c, WS_EINVAL, "null encoder states or cu_frames");
  if (maxF < 1 || maxF > c->d.max_frames) return fail(c, WS_EINVAL, "max_frames_call %d outside 1..%d", maxF, c->d.max_frames);
  if (total_frames < maxF || (int64_t)total_frames > (int64_t)n * maxF)
    return fail(c, WS_EINVAL, "total_frames %d inconsistent with n_req * max_frames_call", total_frames);
  cudaStream_t s = (cudaStream_t)stream;
  return c->d.dtype == WS_BF16 ? cross_kv_impl<bf16>(c, n, req, enc, cu, valid, maxF, total_frames, s)
                               : cross_kv_impl<float>(c, n, req, enc, cu, valid, maxF, total_frames, s);
}

int ws_verify(ws_ctx* c, int n, const int32_t* req, int H, const int32_t* block, const int32_t* blen,
              int32_t* target, float* logits, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (H < 1 || H > c->d.max_block) return fail(c, WS_EINVAL, "H %d outside 1..max_block (%d)", H, c->d.max_block);
  if (!block || !blen || !target) return fail(c, WS_EINVAL, "null block, block_len or target");
  cudaStream_t s = (cudaStream_t)stream;
  return c->d.dtype == WS_BF16 ? verify_impl<bf16>(c, n, req, H, block, blen, target, logits, s)
                               : verify_impl<float>(c, n, req, H, block, blen, target, logits, s);
}

int ws_verify_tree(ws_ctx* c, int n, const int32_t* req, int H, const int32_t* block, const int32_t* blen,
                   int32_t* target, float* logits, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (c->tree_n < 1) return fail(c, WS_EINVAL, "no candidate tree set (ws_set_tree)");
  if (H != c->tree_n) return fail(c, WS_EINVAL, "H %d must equal the tree's row count %d", H, c->tree_n);
  if (!block || !blen || !target) return fail(c, WS_EINVAL, "null block, block_len or target");
  cudaStream_t s = (cudaStream_t)stream;
  const TreeMask tm = c->tree;
  return c->d.dtype == WS_BF16 ? verify_impl<bf16>(c, n, req, H, block, blen, target, logits, s, &tm)
                               : verify_impl<float>(c, n, req, H, block, blen, target, logits, s, &tm);
}

int ws_draft(ws_ctx* c, int n, const int32_t* req, int32_t* block, float temperature, uint64_t seed, uint64_t round,
             float* q_logits, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (c->d.drafter_layers == 0) return fail(c, WS_EUNSUPPORTED, "context has no drafter");
  if (!block) return fail(c, WS_EINVAL, "null block");
  if (!(temperature >= 0.0f)) return fail(c, WS_EINVAL, "temperature must be >= 0");
  if (temperature > 0.0f && !q_logits) return fail(c, WS_EINVAL, "sampling needs q_logits");
  cudaStream_t s = (cudaStream_t)stream;
  return c->d.dtype == WS_BF16 ? draft_impl<bf16>(c, n, req, block, temperature, seed, round, q_logits, s)
                               : draft_impl<float>(c, n, req, block, temperature, seed, round, q_logits, s);
}

int ws_accept(ws_ctx* c, int n, const int32_t* req, const ws_accept_args* a, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (!a) return fail(c, WS_EINVAL, "null accept args");
  if (n == 0) return WS_OK;
  if (a->mode < WS_ACCEPT_GREEDY || a->mode > WS_ACCEPT_TREE) return fail(c, WS_EINVAL, "unknown accept mode");
  if (a->mode == WS_ACCEPT_TREE && (c->tree_n < 1 || a->H != c->tree_n))
    return fail(c, WS_EINVAL, "tree acceptance needs a tree (ws_set_tree) and H equal to its row count");
  if (a->H < 1 || a->H > c->d.max_block) return fail(c, WS_EINVAL, "H outside 1..max_block");
  if (!a->block || !a->block_len || !a->budget || !a->done || !a->n_acc || !a->n_emit || !a->next_block ||
      !a->next_len)
    return fail(c, WS_EINVAL, "null required accept array");
  if (a->next_stride < 1) return fail(c, WS_EINVAL, "next_stride must be >= 1");
  if (a->mode != WS_ACCEPT_SAMPLE && !a->target) return fail(c, WS_EINVAL, "greedy/forced acceptance needs target");
  if (a->mode == WS_ACCEPT_SAMPLE) {
    if (!a->p_logits || !a->q_logits) return fail(c, WS_EINVAL, "sampling acceptance needs p_logits and q_logits");
    if (!(a->temperature > 0.0f)) return fail(c, WS_EINVAL, "sampling acceptance needs temperature > 0");
  }
  if (a->transcript && (!a->out_len || a->tcap < 1)) return fail(c, WS_EINVAL, "transcript needs out_len and tcap");
  AcceptParams p;
  p.a = *a;
  p.req_ids = req;
  p.L = c->L;
  p.K = c->d.K;
  p.V = c->d.vocab;
  p.eos = c->d.eos_id;
  p.max_pos = c->d.max_pos;
  p.suppress = c->suppress;
  p.status = c->status;
  p.pstat = c->pstat;
  p.qstat = c->qstat;
  const bool tree = a->mode == WS_ACCEPT_TREE;
  p.tree_n = tree ? c->tree_n : 0;
  p.parent4 = c->tree_parent4;
  p.tpath = c->tpath;
  if (tree) p.a.mode = WS_ACCEPT_GREEDY;            // the greedy rule, walked over the tree
  CK(launch_accept(n, p, (cudaStream_t)stream, c->cur_pdl));
  if (tree) {
    TreeCommit t;
    t.req_ids = req; t.tpath = c->tpath; t.kv = c->kv; t.kv_layer_bytes = c->kv_layer_bytes;
    t.ptab = c->ptab; t.ppr = c->ppr; t.heads = c->heads; t.es = c->es; t.n_layers = c->d.n_layers;
    const bool hist = c->d.drafter_layers > 0 && c->d.n_hist > 0;
    t.hist = hist ? c->hist : nullptr; t.max_block = c->d.max_block; t.hist_w = hist ? c->d.n_hist * c->d.d_model : 0;
    t.qread = c->readout_layer >= 0 ? (char*)c->qread : nullptr; t.H = a->H; t.d = c->d.d_model;
    CK(launch_tree_commit(n, t, (cudaStream_t)stream, c->cur_pdl));
  }
  return WS_OK;
}

int ws_draft_synthetic(ws_ctx* c, int n, const int32_t* req, int32_t* block, const int32_t* traj, int tlen,
                       const uint8_t* cmask, const int32_t* ctok, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (!block || !traj || !cmask || !ctok || tlen < 1) return fail(c, WS_EINVAL, "null synthetic-draft input");
  CK(launch_draft_synth(n, c->d.K, req, c->L, block, traj, tlen, cmask, ctok, c->d.max_pos, (cudaStream_t)stream,
                        c->cur_pdl));
  return WS_OK;
}

int ws_draft_limit(ws_ctx* c, int n, const int32_t* req, const int32_t* block, int stride_in, const float* q_logits,
                   int k_verify, float threshold, float temperature, int32_t* block_out, int stride_out,
                   int32_t* block_len, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (!block || !block_out || !block_len) return fail(c, WS_EINVAL, "null block, block_out or block_len");
  if (k_verify < 0 || k_verify > c->d.K) return fail(c, WS_EINVAL, "k_verify %d outside 0..K (%d)", k_verify, c->d.K);
  if (stride_in < c->d.K + 1 || stride_out < k_verify + 1)
    return fail(c, WS_EINVAL, "block strides must hold K+1 (in) and k_verify+1 (out) tokens");
  if (!(threshold == threshold) || !(temperature >= 0.0f)) return fail(c, WS_EINVAL, "bad threshold or temperature");
  if (threshold > 0.0f && !q_logits) return fail(c, WS_EINVAL, "a confidence threshold needs q_logits");
  CK(launch_draft_limit(n, c->d.K, block, stride_in, q_logits, c->d.vocab, temperature > 0.0f ? temperature : 1.0f,
                        c->suppress, c->conf, k_verify, threshold, block_out, stride_out, block_len,
                        (cudaStream_t)stream, c->cur_pdl));
  return WS_OK;
}

int ws_set_tree(ws_ctx* c, int n_nodes, const int32_t* parent, const int32_t* rank) {
  if (!c) return fail(nullptr, WS_EINVAL, "null context");
  if (n_nodes == 0) {
    c->tree_n = 0;
    c->tree = linear_tree();
    c->tree_parent4 = c->tree_rank4 = 0;
    return WS_OK;
  }
  if (n_nodes < 1 || n_nodes > c->d.max_block || n_nodes > 16)
    return fail(c, WS_EINVAL, "n_nodes %d outside 0..max_block (%d)", n_nodes, c->d.max_block);
  if (!parent || !rank) return fail(c, WS_EINVAL, "null parent or rank");
  if (parent[0] != -1 || rank[0] != 0) return fail(c, WS_EINVAL, "row 0 is the root: parent -1, rank 0");
  TreeMask t;
  t.depth4 = 0;
  unsigned long long p4 = 0, r4 = 0;
  int depth[16] = {0};
  t.anc[0] = 1u;
  for (int j = 1; j < n_nodes; ++j) {
    if (parent[j] < 0 || parent[j] >= j) return fail(c, WS_EINVAL, "parent[%d] = %d not in 0..%d", j, parent[j], j - 1);
    if (rank[j] < 0 || rank[j] > 15) return fail(c, WS_EINVAL, "rank[%d] = %d outside 0..15", j, rank[j]);
    depth[j] = depth[parent[j]] + 1;
    if (c->d.drafter_layers > 0 && depth[j] > c->d.K)
      return fail(c, WS_EINVAL, "row %d at depth %d beyond the drafter's K = %d rows", j, depth[j], c->d.K);
    t.anc[j] = t.anc[parent[j]] | (1u << j);
    t.depth4 |= (unsigned long long)depth[j] << (4 * j);
    p4 |= (unsigned long long)parent[j] << (4 * j);
    r4 |= (unsigned long long)rank[j] << (4 * j);
  }
  for (int j = n_nodes; j < 16; ++j) t.anc[j] = 0u;
  c->tree_n = n_nodes;
  c->tree = t;
  c->tree_parent4 = p4;
  c->tree_rank4 = r4;
  return WS_OK;
}

int ws_tree_tokens(ws_ctx* c, int n, const int32_t* req, const int32_t* block, int stride_in, const float* q_logits,
                   int32_t* block_out, int stride_out, int32_t* block_len, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (c->tree_n < 1) return fail(c, WS_EINVAL, "no candidate tree set (ws_set_tree)");
  if (!block || !q_logits || !block_out || !block_len) return fail(c, WS_EINVAL, "null block, q_logits, block_out or block_len");
  if (stride_in < 1 || stride_out < c->tree_n) return fail(c, WS_EINVAL, "stride_out must hold the tree's rows");
  for (int j = 1; j < c->tree_n; ++j)
    if (tree_depth(c->tree.depth4, j) > c->d.K) return fail(c, WS_EINVAL, "tree deeper than the K draft rows");
  CK(launch_tree_tokens(n, c->tree_n, c->tree.depth4, c->tree_rank4, req, c->L, c->d.max_pos, block, stride_in,
                        q_logits, c->d.K, c->d.vocab, block_out, stride_out, block_len, (cudaStream_t)stream,
                        c->cur_pdl));
  return WS_OK;
}

int ws_set_readout(ws_ctx* c, int layer, int half_width) {
  if (!c) return fail(nullptr, WS_EINVAL, "null context");
  if (layer < -1 || layer >= c->d.n_layers) return fail(c, WS_EINVAL, "readout layer %d outside -1..n_layers-1", layer);
  if (half_width < 0) return fail(c, WS_EINVAL, "half_width must be >= 0");
  if (half_width > 0 && c->d.drafter_layers == 0) return fail(c, WS_EUNSUPPORTED, "context has no drafter");
  c->readout_layer = layer;
  c->half_width = half_width;
  return WS_OK;
}

int ws_readout(ws_ctx* c, int n, const int32_t* req, const int32_t* row, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (!row) return fail(c, WS_EINVAL, "null row");
  if (c->readout_layer < 0 || c->read_H < 1) return fail(c, WS_EINVAL, "no readout layer set, or no verify since");
  const cudaStream_t s = (cudaStream_t)stream;
  if (c->d.dtype == WS_BF16)
    CK(launch_readout<bf16>(n, c->read_H, req, row, (const bf16*)c->qread, c->d.d_model, xkv_of(c), c->readout_layer,
                            c->Fv, c->d.max_frames, c->rsc, c->rst, c->xcenter, s, c->cur_pdl));
  else
    CK(launch_readout<float>(n, c->read_H, req, row, (const float*)c->qread, c->d.d_model, xkv_of(c),
                             c->readout_layer, c->Fv, c->d.max_frames, c->rsc, c->rst, c->xcenter, s, c->cur_pdl));
  return WS_OK;
}

int ws_get_centers(ws_ctx* c, int n, const int32_t* req, int32_t* out, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (!out) return fail(c, WS_EINVAL, "null output");
  CK(launch_get_lengths(n, req, c->xcenter, out, (cudaStream_t)stream));
  return WS_OK;
}

int ws_sample(ws_ctx* c, int n, const int32_t* req, const float* logits, int rows, float temperature, uint64_t seed,
              uint64_t round, int32_t* out, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (!logits || !out || rows < 1) return fail(c, WS_EINVAL, "null logits/out or rows < 1");
  if (!(temperature > 0.0f)) return fail(c, WS_EINVAL, "temperature must be > 0");
  CK(launch_sample_rows(n, rows, req, logits, c->d.vocab, c->d.vocab, temperature, seed, round, c->suppress, out,
                        rows, 0, (cudaStream_t)stream, c->cur_pdl));
  return WS_OK;
}

int ws_set_suppress(ws_ctx* c, const uint32_t* mask) {
  if (!c) return fail(nullptr, WS_EINVAL, "null context");
  c->suppress = mask;
  return WS_OK;
}

int ws_get_lengths(ws_ctx* c, int n, const int32_t* req, int32_t* out, ws_stream stream) {
  if (int r = check_common(c, n, req, stream)) return r;
  if (n == 0) return WS_OK;
  if (!out) return fail(c, WS_EINVAL, "null output");
  CK(launch_get_lengths(n, req, c->L, out, (cudaStream_t)stream));
  return WS_OK;
}

int ws_status(ws_ctx* c, ws_stream stream, int32_t* host_status) {
  if (!c) return fail(nullptr, WS_EINVAL, "null context");
  cudaStream_t s = (cudaStream_t)stream;
  int32_t v = 0;
  CK(cudaMemcpyAsync(&v, c->status, 4, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  CK(cudaMemsetAsync(c->status, 0, 4, s));
  CK(cudaStreamSynchronize(s));
  if (host_status) *host_status = v;
  if (v) return fail(c, WS_EDEVICE, "device status 0x%x (1 = position >= max_pos, 2 = token id, 4 = frames)", v);
  return WS_OK;
}

const char* ws_gemm_engine(const ws_ctx* c) {
  if (!c) return "none";
  return c->engine == WS_GEMM_TC ? "tcgen05" : "simt";
}

int ws_fused_verify(ws_ctx* c, int enable) {
  if (!c) return fail(nullptr, WS_EINVAL, "null context");
  if (enable >= 0) c->flow_on = enable != 0;
  return (c->flow_ok && c->flow_on) ? 1 : 0;
}

int ws_fused_layernorm(ws_ctx* c, int enable) {
  if (!c) return fail(nullptr, WS_EINVAL, "null context");
  if (enable >= 0) c->ln_in_gemm = enable != 0;
  return c->ln_in_gemm ? 1 : 0;
}

unsigned long long ws_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int ws_capture_begin(ws_ctx* c, ws_stream stream) {
  if (!c) return fail(nullptr, WS_EINVAL, "null context");
  if (!stream) return fail(c, WS_EINVAL, "capture needs a created stream");
  CK(cudaStreamBeginCapture((cudaStream_t)stream, cudaStreamCaptureModeThreadLocal));
  c->cap_start = g_launches.load();
  return WS_OK;
}

int ws_capture_end(ws_ctx* c, ws_stream stream, ws_graph** out) {
  if (!c || !out) return fail(c, WS_EINVAL, "null context or output");
  *out = nullptr;
  cudaGraph_t g = nullptr;
  // kernels recorded while capturing did not run: move them to the graph
  const unsigned long long recorded = g_launches.load() - c->cap_start;
  g_launches.fetch_sub(recorded);
  CK(cudaStreamEndCapture((cudaStream_t)stream, &g));
  cudaGraphExec_t ex = nullptr;
  cudaError_t e = cudaGraphInstantiate(&ex, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return fail(c, WS_ECUDA, "graph instantiate: %s", cudaGetErrorString(e));
  *out = new ws_graph{ex, recorded};
  return WS_OK;
}

int ws_graph_launch(ws_graph* graph, ws_stream stream) {
  if (!graph) return fail(nullptr, WS_EINVAL, "null graph");
  cudaError_t e = cudaGraphLaunch(graph->exec, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(nullptr, WS_ECUDA, "graph launch: %s", cudaGetErrorString(e));
  g_launches.fetch_add(graph->kernels);
  return WS_OK;
}

void ws_graph_free(ws_graph* graph) {
  if (!graph) return;
  cudaGraphExecDestroy(graph->exec);
  delete graph;
}

const char* ws_last_error(const ws_ctx* c) { return c ? c->err.c_str() : g_err.c_str(); }

void ws_free(ws_ctx* c) { delete c; }

}  // extern "C"
