// Internal declarations shared by the CUDA translation units of libws.
// Nothing here is part of the public ABI (include/ws.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/ws.h"

typedef __nv_bfloat16 bf16;

#define WS_DH 64          // head width (Whisper: d_model / n_heads = 64)
#define WS_PAGE 64        // tokens per KV-cache page
#define WS_XCHUNK 64      // keys (frames, cache positions) per attention split

// Device status bits (ws_status).
#define WS_ST_POS 1       // a position at or beyond max_pos was requested
#define WS_ST_TOKEN 2     // a token id outside [0, V) was seen
#define WS_ST_FRAMES 4    // frame counts inconsistent with max_frames

// ------------------------------------------------------------------ conversions
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float gelu_erf(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}

// Total order on floats as unsigned ints (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_order(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Argmax key: value first, then the LOWEST id wins ties.  -0 and +0 are
// equal values, so -0 is keyed as +0 and the tie goes to the lower id.
__device__ __forceinline__ unsigned long long argmax_key(float v, int id) {
  if (v == 0.0f) v = 0.0f;
  return ((unsigned long long)f32_order(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ int argmax_key_id(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

// ------------------------------------------------------------------ Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11): 10 rounds of the Philox S-box with the published multipliers and
// Weyl key increments.
struct Philox4 { uint32_t x[4]; };
__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += 0x9E3779B9u; k1 += 0xBB67AE85u;
  }
  Philox4 o; o.x[0] = c0; o.x[1] = c1; o.x[2] = c2; o.x[3] = c3;
  return o;
}
// The method's uniform in [0,1): counter (slot, round, j, purpose), key = seed.
__device__ __forceinline__ float ws_uniform(uint64_t seed, uint32_t slot, uint64_t rnd, uint32_t j,
                                            uint32_t purpose) {
  Philox4 o = philox4x32_10(slot, (uint32_t)rnd, j, purpose, (uint32_t)seed, (uint32_t)(seed >> 32));
  return (float)(o.x[0] >> 8) * (1.0f / 16777216.0f);
}

// ------------------------------------------------------------------ warp / block reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------------ layer norm of one row
// One warp normalises one row of d fp32 values (d a multiple of 128, at most
// 128 * MAXV): lane l owns the float4 groups at 4*l + 128*i.  Mean and
// variance are per-lane sequential sums followed by a fixed shuffle tree, so
// a row's values never depend on which other rows share the launch.
// ln_rows_warp takes NR rows at once: the loads of all of them are issued
// before any is reduced (one memory round trip for NR rows), and the rows'
// reductions are interleaved phase by phase (their shuffle chains overlap);
// each row's arithmetic is the same as alone.  out(r, k, ...) receives the
// four normalised values of group k of row r.  CG: read x from L2 (rows
// written by other SMs in the same kernel).  Only features k_lo <= k < k_hi
// are normalised and passed to out (the statistics always cover the whole
// row); gain and bias of feature k are read at g[k - g_off], b[k - g_off].
template <bool CG, int NR, int MAXV, class Out>
__device__ __forceinline__ void ln_rows_warp(const float* const* xs, int nr, int d, const void* g, const void* b,
                                             bool g_bf16, Out out, int k_lo = 0, int k_hi = 1 << 30,
                                             int g_off = 0) {
  const int lane = threadIdx.x & 31;
  const int nv = d >> 7;
  float4 v[NR][MAXV];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    if (r < nr) {
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        if (i < nv) {
          const float4* src = reinterpret_cast<const float4*>(xs[r] + 4 * lane + 128 * i);
          v[r][i] = CG ? __ldcg(src) : *src;
        }
      }
    }
  }
  // One row (the layer-norm kernel): gains and biases of this lane's groups
  // are loaded while the reductions run and all before the first output is
  // written, since out stores to global memory the compiler cannot tell
  // apart from g and b (each group's loads would otherwise wait behind the
  // previous stores).  Several rows (a GEMM normalising its operand from
  // shared memory): loaded per group, which keeps the registers down.
  constexpr bool HOIST = NR == 1;
  uint2 gq[MAXV], bq[MAXV];
  float4 gf[MAXV], bf[MAXV];
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int k = 4 * lane + 128 * i;
    if (HOIST && i < nv && k >= k_lo && k < k_hi) {
      if (g_bf16) {
        gq[i] = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(g) + (k - g_off));
        bq[i] = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(b) + (k - g_off));
      } else {
        gf[i] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(g) + (k - g_off));
        bf[i] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(b) + (k - g_off));
      }
    }
  }
  float mean[NR], rstd[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float s = 0.0f;
    if (r < nr) {
#pragma unroll
      for (int i = 0; i < MAXV; ++i)
        if (i < nv) s += (v[r][i].x + v[r][i].y) + (v[r][i].z + v[r][i].w);
    }
    mean[r] = s;
  }
#pragma unroll
  for (int r = 0; r < NR; ++r)
    if (r < nr) mean[r] = warp_sum(mean[r]) / (float)d;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float q = 0.0f;
    if (r < nr) {
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        if (i < nv) {
          const float a = v[r][i].x - mean[r], bb = v[r][i].y - mean[r], c = v[r][i].z - mean[r],
                      e = v[r][i].w - mean[r];
          q += (a * a + bb * bb) + (c * c + e * e);
        }
      }
    }
    rstd[r] = q;
  }
#pragma unroll
  for (int r = 0; r < NR; ++r)
    if (r < nr) rstd[r] = rsqrtf(warp_sum(rstd[r]) / (float)d + 1e-5f);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int k = 4 * lane + 128 * i;
    if (i < nv && k >= k_lo && k < k_hi) {
      float gg[4], bv[4];
      if (!HOIST) {
        if (g_bf16) {
          gq[i] = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(g) + (k - g_off));
          bq[i] = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(b) + (k - g_off));
        } else {
          gf[i] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(g) + (k - g_off));
          bf[i] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(b) + (k - g_off));
        }
      }
      if (g_bf16) {
        const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gq[i].x));
        const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gq[i].y));
        const float2 b01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bq[i].x));
        const float2 b23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bq[i].y));
        gg[0] = g01.x; gg[1] = g01.y; gg[2] = g23.x; gg[3] = g23.y;
        bv[0] = b01.x; bv[1] = b01.y; bv[2] = b23.x; bv[3] = b23.y;
      } else {
        gg[0] = gf[i].x; gg[1] = gf[i].y; gg[2] = gf[i].z; gg[3] = gf[i].w;
        bv[0] = bf[i].x; bv[1] = bf[i].y; bv[2] = bf[i].z; bv[3] = bf[i].w;
      }
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (r < nr)
          out(r, k, (v[r][i].x - mean[r]) * rstd[r] * gg[0] + bv[0], (v[r][i].y - mean[r]) * rstd[r] * gg[1] + bv[1],
              (v[r][i].z - mean[r]) * rstd[r] * gg[2] + bv[2], (v[r][i].w - mean[r]) * rstd[r] * gg[3] + bv[3]);
      }
    }
  }
}

template <bool CG = false, int MAXV = 16, class Out>
__device__ __forceinline__ void ln_row_warp(const float* x, int d, const void* g, const void* b, bool g_bf16,
                                            Out out) {
  const float* xs[1] = {x};
  ln_rows_warp<CG, 1, MAXV>(xs, 1, d, g, b, g_bf16,
                          [&](int, int k, float v0, float v1, float v2, float v3) { out(k, v0, v1, v2, v3); });
}

// ------------------------------------------------------------------ PDL
// Programmatic dependent launch: a kernel may start while its predecessor on
// the stream drains; it must wait before touching the predecessor's outputs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ row maps
// How a row of an activation matrix maps to (request slot, block row j,
// absolute position).  Rows are laid out request-major: r = i * H + j.
enum RowMode { ROW_VERIFY = 0, ROW_DRAFT = 1, ROW_HIST = 2, ROW_PLAIN = 3 };
struct RowMap {
  int mode;
  int H;                       // rows per request in this call
  int max_pos;
  const int32_t* req_ids;      // [n]
  const int32_t* L;            // [max_batch] cache lengths (ctx state)
  const int32_t* block_len;    // [n] (ROW_VERIFY)
  const int32_t* pend_start;   // [max_batch] (ROW_HIST)
  const int32_t* pend_n;       // [max_batch] (ROW_HIST)
};
// A block of verification rows as a candidate tree (Alignment Drift App. E.3):
// row j is embedded at position L + depth(j) and its self-attention sees the
// cache before L and the block rows in anc[j] (bit m = row m, row j itself
// included); its keys and values are stored at cache slot L + j.  The
// linear block is the chain depth(j) = j, anc[j] = rows 0..j.
struct TreeMask {
  unsigned long long depth4;   // depth of row j in bits 4j .. 4j + 3
  uint32_t anc[16];
};
inline TreeMask linear_tree() {
  TreeMask t;
  t.depth4 = 0xFEDCBA9876543210ull;
  for (int j = 0; j < 16; ++j) t.anc[j] = (2u << j) - 1u;
  return t;
}
__host__ __device__ __forceinline__ int tree_depth(unsigned long long depth4, int j) {
  return (int)((depth4 >> (4 * j)) & 15ull);
}
// anc[j] without a dynamic index into the (parameter-space) array
__device__ __forceinline__ uint32_t tree_anc(const TreeMask& t, int j) {
  uint32_t r = 0u;
#pragma unroll
  for (int m = 0; m < 16; ++m) r = (m == j) ? t.anc[m] : r;
  return r;
}

// Returns true when the row holds a real token whose K/V may be written.
__device__ __forceinline__ bool row_info(const RowMap& m, int r, int& slot, int& j, int& pos) {
  int i = r / m.H;
  j = r - i * m.H;
  slot = m.req_ids[i];
  bool valid;
  if (m.mode == ROW_HIST) {
    pos = m.pend_start[slot] + j;
    valid = j < m.pend_n[slot];
  } else {
    pos = m.L[slot] + j;
    valid = (m.mode == ROW_VERIFY) ? (j < m.block_len[i]) : true;
  }
  return valid && pos < m.max_pos;
}

// ------------------------------------------------------------------ KV layouts
// Self / history KV pool of one layer: [n_pages][2 (K,V)][heads][WS_PAGE][64].
// Page of (slot, pos) = ptab[slot * ppr + pos / WS_PAGE].
struct KVPool {
  void* base;                  // this layer's pool
  const int32_t* ptab;
  int ppr;                     // pages per request
  int n_heads;
};
template <typename T>
__device__ __forceinline__ T* kv_ptr(const KVPool& p, int slot, int pos, int kv, int head) {
  int page = p.ptab[slot * p.ppr + pos / WS_PAGE];
  size_t off = (((size_t)page * 2 + kv) * p.n_heads + head) * (WS_PAGE * WS_DH) + (size_t)(pos % WS_PAGE) * WS_DH;
  return reinterpret_cast<T*>(p.base) + off;
}

// Cross (acoustic) K/V of one request and one layer: [2][heads][max_frames][64].
struct XKV {
  void* base;                  // slot 0, layer 0
  size_t slot_stride;          // elements between slots
  size_t layer_stride;         // elements between layers (= 2 * heads * max_frames * 64)
  int max_frames;
  int n_heads;
};
template <typename T>
__device__ __forceinline__ T* xkv_ptr(const XKV& x, int slot, int layer, int kv, int head, int frame) {
  return reinterpret_cast<T*>(x.base) + (size_t)slot * x.slot_stride + (size_t)layer * x.layer_stride +
         ((size_t)kv * x.n_heads + head) * ((size_t)x.max_frames * WS_DH) + (size_t)frame * WS_DH;
}

// ------------------------------------------------------------------ GEMM epilogues
enum EpiKind {
  EPI_STORE = 0,    // out[r, n] = act(y + b)
  EPI_GELU = 1,     // out[r, n] = act(gelu(y + b))
  EPI_F32 = 2,      // outf[r, n] = y + b
  EPI_RESID = 3,    // resid[r, n] += y + b  (+ optional history copy)
  EPI_QKV = 4,      // target self-attention: q -> qout, k/v -> paged cache
  EPI_QKV_DRAFT = 5,// drafter block: RoPE(q) -> qout, RoPE(k) -> kout, v -> vout
  EPI_HISTKV = 6,   // drafter history: RoPE(k), v + b -> history cache
  EPI_CROSSKV = 7,  // acoustic K/V -> per-request slabs
  EPI_LOGITS = 8    // logits (+ suppression) -> optional store + argmax keys
};

struct Epi {
  int kind;
  int d;                        // model width (QKV splits)
  const void* bias;             // [N] model dtype or NULL (QKV: b_q)
  const void* bias2;            // QKV: b_v ; HISTKV: b_v
  void* out; int ldo;           // model-dtype or f32 output
  float* resid; int ldr;
  // history copy of the updated residual (verify, history layers):
  // hist[(slot * max_block + j) * n_hist + hidx][n]
  float* hist; int hist_idx; int n_hist; int max_block;
  RowMap rm;
  KVPool kv;                    // QKV / HISTKV target
  void* kout; void* vout;       // QKV_DRAFT
  const float* rope;            // [max_pos][32][2] (cos, sin) or NULL
  XKV xkv; int xlayer;          // CROSSKV
  const int32_t* cu_frames;     // CROSSKV: [n+1]
  const int32_t* req_ids;       // CROSSKV
  float* logits; long long ldl; // LOGITS
  unsigned long long* amax;     // LOGITS: [M] argmax keys
  const uint32_t* suppress;     // LOGITS
  int32_t* status;
};

// ------------------------------------------------------------------ launchers
// Every kernel launch made by the library is counted (ws_launch_count).
void ws_count_launches(int n);
// Message returned by ws_last_error(NULL) on the calling thread.
void ws_set_thread_error(const char* msg);

// Implemented in ws_gemm_simt.cu / ws_gemm_tc.cu / ws_kernels.cu / ws_attn.cu.
struct GemmShape {
  const void* X; int ldx;       // [M, K] activations, model dtype
  const void* W; int ldw;       // [N, K] weights, model dtype
  int M, N, K;
  int batch;                    // grid.z repeats (CROSSKV: n_req), row offset by cu_frames
  // tcgen05 engine only: X = LayerNorm(ln_x; ln_g, ln_b) computed inside the
  // GEMM (rows of ln_x K floats apart) when tc_ln_input_ok; X is then unused
  const float* ln_x = nullptr;
  const void* ln_g = nullptr;
  const void* ln_b = nullptr;
};

template <typename T> cudaError_t launch_gemm_simt(const GemmShape& g, const Epi& e, cudaStream_t s, bool pdl);

struct TcMap;
// Attention partials and the per-(request, head) arrival counters.  For the
// tensor-core attention (bf16): TMA maps of the acoustic K/V slabs and of
// the target self K/V pool as [rows, 64] bf16 matrices (64 x 64 boxes,
// 128-byte swizzle); kv_base is the pool's row 0.
struct AttnScratch {
  float* part;            // [rows][heads][splits][66]
  int* counters;          // [max_batch][heads], zero between launches
  int32_t* status;
  const TcMap* xkv_map = nullptr;
  const TcMap* kv_map = nullptr;
  const void* kv_base = nullptr;
};

// tcgen05 engine (ws_gemm_tc.cu).  TcMap holds an encoded TMA tensor map.
struct alignas(64) TcMap { unsigned char bytes[128]; };
bool tc_engine_available();
bool tc_encode_map(TcMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
bool tc_encode_rows_f32(TcMap* m, const float* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
int tc_pick_bn(int M, int N, int batch);
// Whether a GEMM of this shape and split-K factor can take its layer-norm
// input in-kernel (GemmShape::ln_x): one 16-token tile, split K, every CTA's
// k-blocks in its ring at once, K a multiple of 128 up to 1280.
bool tc_ln_input_ok(int M, int N, int K, int splits);
// X is the row-major activation buffer [x_rows, K] (bf16); W's map has 128-row boxes.
// mx_cached: the activation map for this call's token tile (tc_pick_bn), or
// NULL to encode one from x_base / x_rows.
cudaError_t launch_gemm_tc(const GemmShape& g, const Epi& e, const TcMap& mw, const TcMap* mx_cached,
                           const void* x_base, uint64_t x_rows, int splits, cudaStream_t s,
                           bool pdl);
cudaError_t tc_init_attributes();
int tc_bn_index(int bn);   // 16,32,64,128,256 -> 0..4
#define WS_ST_TIMEOUT 8   // a bounded wait inside a kernel ran out

template <typename T>
cudaError_t launch_layernorm(int M, int d, const float* x, int ldx, const T* g, const T* b, T* y, int ldy,
                             int group_skip, cudaStream_t s, bool pdl);
template <typename T>
cudaError_t launch_embed_target(int n, int H, const RowMap& rm, unsigned long long depth4, const int32_t* block,
                                const T* E, const T* P, int d, int V, float* x, int32_t* pend_start,
                                int32_t* pend_n, int32_t* status, cudaStream_t s, bool pdl);
template <typename T>
cudaError_t launch_embed_draft(int n, int K1, const int32_t* req_ids, const int32_t* block, const T* E,
                               const T* m, int d, int V, float* x, int32_t* pend_n, int32_t* status,
                               cudaStream_t s, bool pdl);
cudaError_t launch_argmax_init(int M, unsigned long long* keys, cudaStream_t s, bool pdl);
cudaError_t launch_argmax_finalize(int n, int H, const int32_t* block_len, const unsigned long long* keys,
                                   int32_t* out, int out_stride, int out_col0, cudaStream_t s, bool pdl);
template <typename T>
cudaError_t launch_hist_gather(int n, int Hp, const int32_t* req_ids, const int32_t* pend_n,
                               const float* hist, int max_block, int n_hist, int d, T* feat,
                               cudaStream_t s, bool pdl);
template <typename T>
cudaError_t launch_self_attn(int n, int H, const RowMap& rm, const TreeMask& tree, const T* Q, const KVPool& kv,
                             T* O, int n_heads, const AttnScratch& sc, cudaStream_t s, bool pdl);
template <typename T>
cudaError_t launch_draft_attn(int n, int K1, const int32_t* req_ids, const int32_t* L, const T* Q,
                              const T* Kb, const T* Vb, const KVPool& hkv, T* O, int n_heads,
                              int max_pos, const AttnScratch& sc, cudaStream_t s, bool pdl);
template <typename T>
cudaError_t launch_cross_attn(int n, int H, const int32_t* req_ids, const int32_t* Fv, const T* Q,
                              const XKV& x, int layer, T* O, int n_heads, int max_frames_seen,
                              const AttnScratch& sc, cudaStream_t s, bool pdl);
template <typename T>
cudaError_t attn_init_attributes();
cudaError_t launch_rope_table(float* tab, int max_pos, cudaStream_t s);
cudaError_t launch_set_frames(int n, const int32_t* req_ids, const int32_t* cu, const int32_t* valid,
                              int max_frames, int32_t* Fc, int32_t* Fv, int32_t* status, cudaStream_t s);
cudaError_t launch_reset(int n, const int32_t* req_ids, int32_t* L, int32_t* pend_n, int32_t* xcenter,
                         cudaStream_t s);
template <typename T>
cudaError_t launch_readout(int n, int H, const int32_t* req_ids, const int32_t* row, const T* q, int d, const XKV& x,
                           int layer, const int32_t* Fv, int max_frames, float* sc, float2* st, int32_t* xcenter,
                           cudaStream_t s, bool pdl);
template <typename T>
cudaError_t launch_window_attn(int n, int H, const int32_t* req_ids, const int32_t* Fv, const int32_t* xcenter, int w,
                               const T* Q, int d, const XKV& x, int layer, T* O, cudaStream_t s, bool pdl);
cudaError_t launch_sample_rows(int n, int rows, const int32_t* req_ids, const float* logits, long long row_stride,
                               int V, float T, uint64_t seed, uint64_t rnd, const uint32_t* suppress,
                               int32_t* out, int out_stride, int out_col0, cudaStream_t s, bool pdl);
struct AcceptParams {
  ws_accept_args a;
  const int32_t* req_ids;
  int32_t* L;
  int K, V, eos;
  const uint32_t* suppress;
  int32_t* status;
  float2* pstat;     // sampling: (max, sum exp) of each target row [n][H] at T ...
  float2* qstat;     // ... and of each drafter row [n][K] (filled by launch_accept)
  int max_pos;
  int tree_n;                  // > 0: greedy acceptance walks a candidate tree of this many rows
  unsigned long long parent4;  // tree: parent row of row j in bits 4j .. 4j + 3
  int32_t* tpath;              // tree: per request [L before, a, path rows 0..a] (WS_TREE_REC ints)
};
#define WS_TREE_REC 18
// Move the accepted root path's self keys / values (every target layer),
// history rows and readout queries from their tree rows to block rows 0..a.
struct TreeCommit {
  const int32_t* req_ids;
  const int32_t* tpath;        // written by the acceptance kernel
  char* kv;                    // self K/V pool of layer 0
  size_t kv_layer_bytes;
  const int32_t* ptab;
  int ppr, heads, es, n_layers;
  float* hist;                 // [slot][max_block][hist_w] fp32, or NULL
  int max_block, hist_w;
  char* qread;                 // [n * H][d] model dtype, or NULL
  int H, d;
};
cudaError_t launch_tree_commit(int n, const TreeCommit& t, cudaStream_t s, bool pdl);
// Tokens of a fixed candidate tree from the drafter's logits: row j at
// depth k >= 1 takes the rank(j)-th largest logit of mask row k - 1 (ties
// to the lower id); row 0 keeps the anchor.
cudaError_t launch_tree_tokens(int n, int n_nodes, unsigned long long depth4, unsigned long long rank4,
                               const int32_t* req_ids, const int32_t* L, int max_pos, const int32_t* block,
                               int stride_in, const float* q, int K, int V, int32_t* out, int stride_out,
                               int32_t* blen, cudaStream_t s, bool pdl);
// Sampling acceptance first fills pstat / qstat with one CTA per logits row,
// then runs one CTA per request.
cudaError_t launch_accept(int n, const AcceptParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_draft_synth(int n, int K, const int32_t* req_ids, const int32_t* L, int32_t* block,
                               const int32_t* traj, int tlen, const uint8_t* cmask, const int32_t* ctok,
                               int max_pos, cudaStream_t s, bool pdl);
cudaError_t launch_get_lengths(int n, const int32_t* req_ids, const int32_t* L, int32_t* out, cudaStream_t s);
cudaError_t launch_draft_limit(int n, int K, const int32_t* block, int stride_in, const float* q, int V, float T,
                               const uint32_t* sup, float* conf, int k_verify, float thr, int32_t* out,
                               int stride_out, int32_t* blen, cudaStream_t s, bool pdl);
