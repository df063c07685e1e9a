// Block-verify attention kernels (decode-shaped: up to 16 query rows per
// request and head, keys streamed through shared memory in tiles of 32).
//
// Every query row runs its own online softmax over key tiles that start at
// absolute key 0, with fixed-order warp reductions, so a row's result does
// not depend on how many other rows share the block (block verification and
// one-token decoding give bit-identical rows).
#include "ws_internal.cuh"

namespace {

constexpr int KT = 32;        // keys per tile
constexpr int MAXR = 16;      // rows per request per CTA
constexpr int NW = 4;         // warps per CTA
constexpr int RPW = MAXR / NW;

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t s, bool pdl, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

struct RowState { float m, l, a0, a1; };

__device__ __forceinline__ void row_init(RowState& s) { s.m = -INFINITY; s.l = 0.0f; s.a0 = 0.0f; s.a1 = 0.0f; }

// One tile of keys for one row held by a warp.  nvalid = keys of the tile
// the row may see (prefix of the tile).  q in shared memory [64].
__device__ __forceinline__ void row_tile(RowState& st, const float* q, const float (*Kt)[WS_DH + 1],
                                         const float (*Vt)[WS_DH], int nvalid) {
  const int lane = threadIdx.x & 31;
  float s = -INFINITY;
  if (lane < nvalid) {
    float acc = 0.0f;
#pragma unroll 16
    for (int d = 0; d < WS_DH; ++d) acc = fmaf(q[d], Kt[lane][d], acc);
    s = acc * 0.125f;                       // 1/sqrt(64)
  }
  const float mt = warp_max(s);
  const float mn = fmaxf(st.m, mt);
  const float p = lane < nvalid ? expf(s - mn) : 0.0f;
  const float corr = expf(st.m - mn);
  st.l = st.l * corr + warp_sum(p);
  float a0 = st.a0 * corr, a1 = st.a1 * corr;
  for (int k = 0; k < nvalid; ++k) {
    const float pk = __shfl_sync(0xffffffffu, p, k);
    const float2 v = *reinterpret_cast<const float2*>(&Vt[k][2 * lane]);
    a0 = fmaf(pk, v.x, a0);
    a1 = fmaf(pk, v.y, a1);
  }
  st.a0 = a0; st.a1 = a1; st.m = mn;
}

template <typename T>
__device__ __forceinline__ void load_tile(float (*Kt)[WS_DH + 1], float (*Vt)[WS_DH], const T* kp, const T* vp,
                                          int nkeys) {
  // kp/vp point at key 0 of the tile, rows of 64 contiguous elements
  for (int idx = threadIdx.x; idx < KT * WS_DH; idx += NW * 32) {
    int k = idx / WS_DH, d = idx - k * WS_DH;
    bool ok = k < nkeys;
    Kt[k][d] = ok ? to_f<T>(kp[(size_t)k * WS_DH + d]) : 0.0f;
    Vt[k][d] = ok ? to_f<T>(vp[(size_t)k * WS_DH + d]) : 0.0f;
  }
}

// ------------------------------------------------------------------ target self-attention
// Row j of request i sits at position L + j and sees cache keys 0..L+j
// (causal; the block's own keys were written by the QKV epilogue).
template <typename T>
__global__ void __launch_bounds__(NW * 32) self_attn_kernel(RowMap rm, const T* Q, KVPool kv, T* O, int d) {
  __shared__ float Kt[KT][WS_DH + 1];
  __shared__ __align__(16) float Vt[KT][WS_DH];
  __shared__ float qs[MAXR][WS_DH];
  pdl_wait();
  const int i = blockIdx.x, head = blockIdx.y, H = rm.H;
  const int slot = rm.req_ids[i];
  const int L = rm.L[slot];
  const int nrow = min(rm.block_len[i], H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int idx = threadIdx.x; idx < H * WS_DH; idx += NW * 32) {
    int j = idx / WS_DH, dd = idx - j * WS_DH;
    qs[j][dd] = to_f<T>(Q[((size_t)i * H + j) * d + head * WS_DH + dd]);
  }
  const int nkeys = min(L + nrow, rm.max_pos);
  RowState st[RPW];
#pragma unroll
  for (int u = 0; u < RPW; ++u) row_init(st[u]);
  for (int t0 = 0; t0 < nkeys; t0 += KT) {
    __syncthreads();
    const int pos0 = t0;   // tiles never straddle a page (WS_PAGE % KT == 0)
    load_tile<T>(Kt, Vt, kv_ptr<T>(kv, slot, pos0, 0, head), kv_ptr<T>(kv, slot, pos0, 1, head),
                 min(KT, nkeys - t0));
    __syncthreads();
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      const int j = warp + u * NW;
      if (j >= nrow) continue;
      const int nk = min(L + j + 1, rm.max_pos);     // keys visible to this row
      if (t0 >= nk) continue;
      row_tile(st[u], qs[j], Kt, Vt, min(KT, nk - t0));
    }
  }
  pdl_trigger();
#pragma unroll
  for (int u = 0; u < RPW; ++u) {
    const int j = warp + u * NW;
    if (j >= H) continue;
    float o0 = 0.0f, o1 = 0.0f;
    if (j < nrow && st[u].l > 0.0f) { o0 = st[u].a0 / st[u].l; o1 = st[u].a1 / st[u].l; }
    T* o = O + ((size_t)i * H + j) * d + head * WS_DH + 2 * lane;
    o[0] = from_f<T>(o0);
    o[1] = from_f<T>(o1);
  }
}

// ------------------------------------------------------------------ cross-attention
// Split s covers frames [s*128, (s+1)*128) of the valid frames; partial
// (m, l, acc[64]) per (row, head, split), folded in split order afterwards.
template <typename T>
__global__ void __launch_bounds__(NW * 32) cross_attn_part_kernel(int H, const int32_t* req_ids, const int32_t* Fv,
                                                                  const T* Q, XKV x, int layer, float* part,
                                                                  int d, int n_split) {
  __shared__ float Kt[KT][WS_DH + 1];
  __shared__ __align__(16) float Vt[KT][WS_DH];
  __shared__ float qs[MAXR][WS_DH];
  pdl_wait();
  const int i = blockIdx.x, head = blockIdx.y, sp = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = req_ids[i];
  const int F = Fv[slot];
  const int f0 = sp * WS_XCHUNK, f1 = min(F, f0 + WS_XCHUNK);
  for (int idx = threadIdx.x; idx < H * WS_DH; idx += NW * 32) {
    int j = idx / WS_DH, dd = idx - j * WS_DH;
    qs[j][dd] = to_f<T>(Q[((size_t)i * H + j) * d + head * WS_DH + dd]);
  }
  RowState st[RPW];
#pragma unroll
  for (int u = 0; u < RPW; ++u) row_init(st[u]);
  const T* kb = xkv_ptr<T>(x, slot, layer, 0, head, 0);
  const T* vb = xkv_ptr<T>(x, slot, layer, 1, head, 0);
  for (int t0 = f0; t0 < f1; t0 += KT) {
    __syncthreads();
    const int nk = min(KT, f1 - t0);
    load_tile<T>(Kt, Vt, kb + (size_t)t0 * WS_DH, vb + (size_t)t0 * WS_DH, nk);
    __syncthreads();
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      const int j = warp + u * NW;
      if (j >= H) continue;
      row_tile(st[u], qs[j], Kt, Vt, nk);
    }
  }
  pdl_trigger();
#pragma unroll
  for (int u = 0; u < RPW; ++u) {
    const int j = warp + u * NW;
    if (j >= H) continue;
    float* p = part + ((((size_t)i * H + j) * (d / WS_DH) + head) * n_split + sp) * (WS_DH + 2);
    if (lane == 0) { p[0] = st[u].m; p[1] = st[u].l; }
    p[2 + 2 * lane] = st[u].a0;
    p[3 + 2 * lane] = st[u].a1;
  }
}

template <typename T>
__global__ void __launch_bounds__(128) cross_attn_combine_kernel(int rows, const float* part, T* O, int d,
                                                                 int n_split) {
  pdl_wait();
  const int heads = d / WS_DH;
  const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= rows * heads) return;
  const int r = w / heads, head = w - r * heads;
  const float* p = part + ((size_t)r * heads + head) * n_split * (WS_DH + 2);
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, p[s * (WS_DH + 2)]);
  float den = 0.0f, n0 = 0.0f, n1 = 0.0f;
  for (int s = 0; s < n_split; ++s) {
    const float* q = p + s * (WS_DH + 2);
    if (q[1] <= 0.0f) continue;
    const float c = expf(q[0] - M);
    den = fmaf(q[1], c, den);
    n0 = fmaf(q[2 + 2 * lane], c, n0);
    n1 = fmaf(q[3 + 2 * lane], c, n1);
  }
  pdl_trigger();
  T* o = O + (size_t)r * d + head * WS_DH + 2 * lane;
  o[0] = from_f<T>(den > 0.0f ? n0 / den : 0.0f);
  o[1] = from_f<T>(den > 0.0f ? n1 / den : 0.0f);
}

// ------------------------------------------------------------------ drafter attention
// Block rows of request i attend, in one softmax, to the history keys at
// positions 0..t-1 (t = L, the anchor position) and to all K+1 block keys:
// bidirectional inside the block (Whisper-Flash §3.2, Appendix A.2).
template <typename T>
__global__ void __launch_bounds__(NW * 32) draft_attn_kernel(int K1, const int32_t* req_ids, const int32_t* Lp,
                                                             const T* Q, const T* Kb, const T* Vb, KVPool hkv, T* O,
                                                             int d, int max_pos) {
  __shared__ float Kt[KT][WS_DH + 1];
  __shared__ __align__(16) float Vt[KT][WS_DH];
  __shared__ float qs[MAXR][WS_DH];
  pdl_wait();
  const int i = blockIdx.x, head = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = req_ids[i];
  const int t = min(Lp[slot], max_pos);
  for (int idx = threadIdx.x; idx < K1 * WS_DH; idx += NW * 32) {
    int j = idx / WS_DH, dd = idx - j * WS_DH;
    qs[j][dd] = to_f<T>(Q[((size_t)i * K1 + j) * d + head * WS_DH + dd]);
  }
  RowState st[RPW];
#pragma unroll
  for (int u = 0; u < RPW; ++u) row_init(st[u]);
  for (int t0 = 0; t0 < t; t0 += KT) {
    __syncthreads();
    const int nk = min(KT, t - t0);
    load_tile<T>(Kt, Vt, kv_ptr<T>(hkv, slot, t0, 0, head), kv_ptr<T>(hkv, slot, t0, 1, head), nk);
    __syncthreads();
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      const int j = warp + u * NW;
      if (j < K1) row_tile(st[u], qs[j], Kt, Vt, nk);
    }
  }
  // the block's own keys (rows of Kb / Vb, one row of d per block row)
  __syncthreads();
  for (int idx = threadIdx.x; idx < KT * WS_DH; idx += NW * 32) {
    int k = idx / WS_DH, dd = idx - k * WS_DH;
    bool ok = k < K1;
    Kt[k][dd] = ok ? to_f<T>(Kb[((size_t)i * K1 + k) * d + head * WS_DH + dd]) : 0.0f;
    Vt[k][dd] = ok ? to_f<T>(Vb[((size_t)i * K1 + k) * d + head * WS_DH + dd]) : 0.0f;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < RPW; ++u) {
    const int j = warp + u * NW;
    if (j < K1) row_tile(st[u], qs[j], Kt, Vt, K1);
  }
  pdl_trigger();
#pragma unroll
  for (int u = 0; u < RPW; ++u) {
    const int j = warp + u * NW;
    if (j >= K1) continue;
    T* o = O + ((size_t)i * K1 + j) * d + head * WS_DH + 2 * lane;
    o[0] = from_f<T>(st[u].a0 / st[u].l);
    o[1] = from_f<T>(st[u].a1 / st[u].l);
  }
}

}  // namespace

template <typename T>
cudaError_t launch_self_attn(int n, int H, const RowMap& rm, const T* Q, const KVPool& kv, T* O, int n_heads,
                             cudaStream_t s, bool pdl) {
  if (H > MAXR) return cudaErrorInvalidValue;
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n, n_heads), dim3(NW * 32), s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, self_attn_kernel<T>, rm, Q, kv, O, n_heads * WS_DH);
}

template <typename T>
cudaError_t launch_cross_attn(int n, int H, const int32_t* req_ids, const int32_t* Fv, const T* Q, const XKV& x,
                              int layer, float* part, T* O, int n_heads, int n_split, cudaStream_t s, bool pdl) {
  if (H > MAXR) return cudaErrorInvalidValue;
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n, n_heads, n_split), dim3(NW * 32), s, pdl, at);
  ws_count_launches(1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, cross_attn_part_kernel<T>, H, req_ids, Fv, Q, x, layer, part,
                                     n_heads * WS_DH, n_split);
  if (e != cudaSuccess) return e;
  const int rows = n * H;
  cudaLaunchConfig_t cfg2 = make_cfg(dim3((rows * n_heads + 3) / 4), dim3(128), s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg2, cross_attn_combine_kernel<T>, rows, (const float*)part, O, n_heads * WS_DH,
                            n_split);
}

template <typename T>
cudaError_t launch_draft_attn(int n, int K1, const int32_t* req_ids, const int32_t* L, const T* Q, const T* Kb,
                              const T* Vb, const KVPool& hkv, T* O, int n_heads, int max_pos, cudaStream_t s,
                              bool pdl) {
  if (K1 > MAXR) return cudaErrorInvalidValue;
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n, n_heads), dim3(NW * 32), s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, draft_attn_kernel<T>, K1, req_ids, L, Q, Kb, Vb, hkv, O, n_heads * WS_DH,
                            max_pos);
}

#define INST(T)                                                                                                  \
  template cudaError_t launch_self_attn<T>(int, int, const RowMap&, const T*, const KVPool&, T*, int,            \
                                           cudaStream_t, bool);                                                   \
  template cudaError_t launch_cross_attn<T>(int, int, const int32_t*, const int32_t*, const T*, const XKV&, int, \
                                            float*, T*, int, int, cudaStream_t, bool);                            \
  template cudaError_t launch_draft_attn<T>(int, int, const int32_t*, const int32_t*, const T*, const T*,        \
                                            const T*, const KVPool&, T*, int, int, cudaStream_t, bool);
INST(float)
INST(bf16)
