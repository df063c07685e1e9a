// Decode-shaped attention for block verification and drafting: up to 16
// query rows per request and head against a key range split into 64-key
// chunks.  Each chunk gives a partial (max, sum, 64 weighted values) and
// the partials of a row are folded in chunk order.  Three variants:
//
//   * attn_cluster_kernel (bf16, calls of up to 4 requests): one
//     thread-block cluster per (request, head), one warp per chunk computing
//     its partial with mma.sync; the cluster folds the rows through
//     distributed shared memory.
//   * attn_stream_kernel + attn_fold_kernel (bf16, larger calls): persistent
//     warps stream (request, head, chunk) units through double-buffered TMA
//     slots; a second kernel folds the partials.
//   * attn_split_kernel (fp32 contexts, the drafter's block attention): one
//     CTA per (request, head, split) stages the split with bulk copies and
//     runs a scalar online softmax per row; the CTA that finishes last for a
//     (request, head) folds the partials.
//
// Splits start at absolute key multiples of 64 and every reduction has a
// fixed order, so a row's result does not depend on how many other rows
// share the block: verifying a block and decoding one token at a time give
// bit-identical rows.
#include <cuda.h>
#include <cooperative_groups.h>

#include "ws_attn_common.cuh"
#include "ws_attn_mma.cuh"

namespace {

constexpr int SPLIT = WS_XCHUNK;   // keys per split (64)
constexpr int NW = 8;              // warps per CTA
constexpr int MAXR = 16;           // query rows per request
constexpr int PART = WS_ATTN_PART;
constexpr long long WAIT_BUDGET = 1ll << 32;

enum { MODE_SELF = 0, MODE_CROSS = 1, MODE_DRAFT = 2 };

struct AttnArgs {
  int mode;                  // MODE_SELF / MODE_CROSS / MODE_DRAFT (kernels compiled for any mode)
  int n_req;                 // requests in the call
  int H;                     // query rows per request
  int n_split;               // splits per (request, head); DRAFT: history splits + 1 block split
  int d, max_pos;
  const int32_t* req_ids;
  const int32_t* L;          // cache lengths (SELF: block starts at L; DRAFT: history < L)
  const int32_t* block_len;  // SELF: valid rows per request
  const int32_t* Fv;         // CROSS: valid frames per slot
  const void* Q;             // [n*H, d]
  KVPool kv;                 // SELF / DRAFT history
  XKV x; int xlayer;         // CROSS
  const void* Kb; const void* Vb;   // DRAFT block keys/values [n*H, d]
  float* part;               // [n*H][heads][n_split][PART]
  int* counters;             // [n][heads], zero between launches
  void* O;                   // [n*H, d]
  int32_t* status;
  TreeMask tree;             // SELF: which block rows each row sees
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    if (ok) return true;
    if (clock64() - t0 > WAIT_BUDGET) return false;
  }
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"((uint64_t)src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

template <typename T, int MODE>
__global__ void __launch_bounds__(NW * 32) attn_split_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_last;
  T* Kraw = reinterpret_cast<T*>(dsm);
  T* Vraw = Kraw + SPLIT * WS_DH;
  float (*Kt)[WS_DH + 1] = reinterpret_cast<float (*)[WS_DH + 1]>(Vraw + SPLIT * WS_DH);
  float (*Vt)[WS_DH] = reinterpret_cast<float (*)[WS_DH]>(reinterpret_cast<float*>(Kt) + SPLIT * (WS_DH + 1));
  float (*qs)[WS_DH] = reinterpret_cast<float (*)[WS_DH]>(reinterpret_cast<float*>(Vt) + SPLIT * WS_DH);
  float* pws = reinterpret_cast<float*>(qs) + MAXR * WS_DH;

  const int i = blockIdx.x, head = blockIdx.y, sp = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads = a.d / WS_DH, H = a.H;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();        // the next kernel may launch and run its prologue now
  pdl_wait();

  // ---- which keys this split covers, and how many rows may see them
  const int slot = a.req_ids[i];
  int k_lo = sp * SPLIT, k_hi = k_lo, nrow = H, Lr = 0;
  bool block_split = false;
  if (MODE == MODE_SELF) {
    Lr = a.L[slot];
    nrow = min(a.block_len[i], H);
    k_hi = min(min(Lr + nrow, a.max_pos), k_lo + SPLIT);
  } else if (MODE == MODE_CROSS) {
    k_hi = min(a.Fv[slot], k_lo + SPLIT);
  } else {
    Lr = min(a.L[slot], a.max_pos);
    block_split = sp == a.n_split - 1;
    k_hi = block_split ? k_lo : min(Lr, k_lo + SPLIT);
  }
  const int nk = block_split ? H : max(0, k_hi - k_lo);

  // ---- stage keys and values
  if (nk > 0 && !block_split) {
    if (threadIdx.x == 0) {
      const T *ks, *vs;
      if (MODE == MODE_CROSS) {
        ks = xkv_ptr<T>(a.x, slot, a.xlayer, 0, head, k_lo);
        vs = xkv_ptr<T>(a.x, slot, a.xlayer, 1, head, k_lo);
      } else {
        ks = kv_ptr<T>(a.kv, slot, k_lo, 0, head);
        vs = kv_ptr<T>(a.kv, slot, k_lo, 1, head);
      }
      const uint32_t bytes = (uint32_t)(nk * WS_DH * sizeof(T));
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&bar)), "r"(2 * bytes)
                   : "memory");
      bulk_g2s(Kraw, ks, bytes, &bar);
      bulk_g2s(Vraw, vs, bytes, &bar);
    }
  }
  const T* Q = reinterpret_cast<const T*>(a.Q);
  for (int idx = threadIdx.x; idx < H * WS_DH; idx += NW * 32) {
    const int j = idx / WS_DH, dd = idx - j * WS_DH;
    qs[j][dd] = to_f<T>(Q[((size_t)i * H + j) * a.d + head * WS_DH + dd]);
  }
  bool ok = true;
  if (nk > 0 && !block_split) ok = mbar_wait(&bar, 0);
  if (!ok && threadIdx.x == 0) atomicOr(a.status, WS_ST_TIMEOUT);
  if (nk > 0) {
    for (int idx = threadIdx.x; idx < nk * WS_DH; idx += NW * 32) {
      const int k = idx / WS_DH, dd = idx - k * WS_DH;
      float kv, vv;
      if (block_split) {
        kv = to_f<T>(reinterpret_cast<const T*>(a.Kb)[((size_t)i * H + k) * a.d + head * WS_DH + dd]);
        vv = to_f<T>(reinterpret_cast<const T*>(a.Vb)[((size_t)i * H + k) * a.d + head * WS_DH + dd]);
      } else {
        kv = to_f<T>(Kraw[idx]);
        vv = to_f<T>(Vraw[idx]);
      }
      Kt[k][dd] = kv;
      Vt[k][dd] = vv;
    }
  }
  __syncthreads();

  // ---- one online softmax per row over this split
#pragma unroll
  for (int u = 0; u < MAXR / NW; ++u) {
    const int j = warp + u * NW;
    if (j >= H) continue;
    RowState st;
    st.m = -INFINITY; st.l = 0.f; st.a0 = 0.f; st.a1 = 0.f;
    uint64_t vm = prefix_mask(nk);                      // keys of this split row j may see
    if (MODE == MODE_SELF) vm = (j < nrow) ? self_key_mask(k_lo, k_hi - k_lo, Lr, tree_anc(a.tree, j)) : 0ull;
    const int visible = vm ? 64 - __clzll((long long)vm) : 0;
    for (int k0 = 0; k0 < visible; k0 += 32)
      row_subtile(st, qs[j], Kt, Vt, k0, min(32, visible - k0), pws + warp * 32, (uint32_t)(vm >> k0));
    float* p = a.part + ((((size_t)i * H + j) * heads + head) * a.n_split + sp) * PART;
    if (lane == 0) { p[0] = st.m; p[1] = st.l; }
    p[2 + 2 * lane] = st.a0;
    p[3 + 2 * lane] = st.a1;
  }

  // ---- the last split of (request, head) folds the partials in split order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* c = a.counters + (size_t)i * heads + head;
    const int old = atomicAdd(c, 1);
    s_last = old == a.n_split - 1;
    if (s_last) *c = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  T* O = reinterpret_cast<T*>(a.O);
#pragma unroll
  for (int u = 0; u < MAXR / NW; ++u) {
    const int j = warp + u * NW;
    if (j >= H) continue;
    const float* p = a.part + (((size_t)i * H + j) * heads + head) * a.n_split * PART;
    float o0, o1;
    attn_fold_row<false>(p, a.n_split, o0, o1);
    T* o = O + ((size_t)i * H + j) * a.d + head * WS_DH + 2 * lane;
    o[0] = from_f<T>(o0);
    o[1] = from_f<T>(o1);
  }
}

// ------------------------------------------------------------------ tensor-core variant (bf16)
// K/V chunks of 64 keys arrive by 2-D TMA (64 x 64 bf16 boxes, 128-byte
// swizzle); attn_chunk_partial computes a chunk's partial on tensor cores.
constexpr int CHUNK_BYTES = 2 * WS_XCHUNK * WS_DH * 2;   // K + V, 16 KB

__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ streaming variant
// Persistent warps walk the (request, head, group of 4 chunks) units: global
// warp gw = blockIdx.x * SW + w takes the contiguous range [gw * U / GW,
// (gw + 1) * U / GW) of the U units (GW = all warps), so it streams one
// (request, head)'s chunks in key order and reloads its query fragments only
// when the head changes.  Each warp owns NSLOT 16 KB slots and keeps the K
// and V boxes of its next NSLOT - 1 chunks in flight by TMA while it computes
// the current one (two slots per warp measured faster than four slots with
// half the warps: per-warp compute, not latency, bounds it; seven warps in
// one CTA per SM fill the shared memory); a slot's
// mbarrier has one consumer, which takes its phases in order.  A unit's chunk partials are merged in
// registers and stored once; a second kernel (attn_fold_kernel) folds each
// row's group partials in group order.
constexpr int SW = 7;                        // warps per CTA, one CTA per SM (7 x 32 KB of slots)
constexpr int NSLOT = 2;                     // TMA slots per warp: the next chunk lands while one is computed
constexpr int STREAM_SMEM = SW * NSLOT * CHUNK_BYTES + 1024;
static_assert(STREAM_SMEM <= 227 * 1024, "streaming slots exceed the shared memory of one CTA");

// MODE < 0: the mode is a.mode (one compiled copy serves self- and cross-attention)
template <int MODE>
__device__ __forceinline__ void unit_range(const AttnArgs& a, int i, int sp, int& k_lo, int& nk, int& Lr, int& nrow) {
  const int mode = MODE >= 0 ? MODE : a.mode;
  const int slot = a.req_ids[i];
  k_lo = sp * WS_XCHUNK;
  Lr = 0;
  nrow = a.H;
  int kend;
  if (mode == MODE_SELF) {
    Lr = a.L[slot];
    nrow = min(a.block_len[i], a.H);
    kend = min(Lr + nrow, a.max_pos);
  } else {
    kend = a.Fv[slot];
  }
  nk = max(0, min(kend - k_lo, WS_XCHUNK));
}

// Issue unit u's K and V boxes into dst (lane 0); returns whether bytes were requested.
template <int MODE>
__device__ __forceinline__ bool stage_unit(const AttnArgs& a, const CUtensorMap* map, const bf16* kv_base, int u,
                                           uint8_t* dst, uint64_t* bar) {
  const int mode = MODE >= 0 ? MODE : a.mode;
  const int heads = a.d / WS_DH, ns = a.n_split;
  const int i = u / (heads * ns), head = (u / ns) % heads, sp = u % ns;
  int k_lo, nk, Lr, nrow;
  unit_range<MODE>(a, i, sp, k_lo, nk, Lr, nrow);
  if (nk <= 0) return false;
  const int slot = a.req_ids[i];
  const bf16 *ks, *vs;
  if (mode == MODE_CROSS) {
    ks = xkv_ptr<bf16>(a.x, slot, a.xlayer, 0, head, k_lo);
    vs = xkv_ptr<bf16>(a.x, slot, a.xlayer, 1, head, k_lo);
  } else {
    ks = kv_ptr<bf16>(a.kv, slot, k_lo, 0, head);
    vs = kv_ptr<bf16>(a.kv, slot, k_lo, 1, head);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier reads / writes of the slot first
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(CHUNK_BYTES)
               : "memory");
  tma2d(dst, map, bar, 0, (int)((ks - kv_base) / WS_DH));
  tma2d(dst + CHUNK_BYTES / 2, map, bar, 0, (int)((vs - kv_base) / WS_DH));
  return true;
}

// Chunks per partial of the streaming variant: a warp merges the partials of
// ATTN_GROUP consecutive 64-key chunks of one (request, head) in registers
// (attn_merge, chunk order) and writes one partial per group, which the fold
// kernel folds in group order; the cluster variant groups the same way.
constexpr int STREAM_GROUP = ATTN_GROUP;

template <int MODE>
__global__ void __launch_bounds__(SW * 32) attn_stream_kernel(const __grid_constant__ CUtensorMap tmKV, AttnArgs a,
                                                               const bf16* kv_base) {
  extern __shared__ uint8_t dsm_s[];
  __shared__ __align__(8) uint64_t bar[SW][NSLOT];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_s) + 1023) & ~uintptr_t(1023));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int heads = a.d / WS_DH, H = a.H, ns = a.n_split;
  const int ng = (ns + STREAM_GROUP - 1) / STREAM_GROUP;      // partials per (request, head)
  const int mode = MODE >= 0 ? MODE : a.mode;
  const int total = a.n_req * heads * ng;                     // units: (request, head, group)
  const int gw = blockIdx.x * SW + w, GW = gridDim.x * SW;
  uint8_t* slots = base + w * NSLOT * CHUNK_BYTES;
  if (lane < NSLOT) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[w][lane])) : "memory");
  if (lane == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  pdl_trigger();
  // Acoustic K/V, frame counts and request ids were all written before this
  // library call began (the first kernel of every call releases its
  // dependents only after its own dependency wait), so cross-attention
  // stages its first chunks before waiting on the previous kernel; only the
  // queries depend on it.  Self-attention reads cache rows this call wrote.
  if (mode == MODE_SELF) pdl_wait();
  // The warp walks the chunks of its units [u_beg, u_end) in order; walk
  // chunk k lives in slot k % NSLOT.
  const int u_beg = (int)((long long)gw * total / GW), u_end = (int)((long long)(gw + 1) * total / GW);
  auto sp_first = [&](int u) { return (u % ng) * STREAM_GROUP; };
  auto sp_end = [&](int u) { return min(ns, sp_first(u) + STREAM_GROUP); };
  auto flat = [&](int u, int sp) { return (u / ng) * ns + sp; };     // (request, head) * ns + chunk
  // loaded[b]: slot b holds a requested, not yet consumed copy; uses[b]: phases consumed on bar[w][b]
  bool loaded[NSLOT];
  uint32_t uses[NSLOT];
#pragma unroll
  for (int b = 0; b < NSLOT; ++b) { loaded[b] = false; uses[b] = 0u; }
  int lu = u_beg, lsp = u_beg < u_end ? sp_first(u_beg) : 0, staged = 0;   // next walk chunk to stage
  auto stage_next = [&]() {
    if (lu >= u_end) return;
    const int sl = staged % NSLOT;
    bool ok = false;
    if (lane == 0) ok = stage_unit<MODE>(a, &tmKV, kv_base, flat(lu, lsp), slots + sl * CHUNK_BYTES, &bar[w][sl]);
    ok = __shfl_sync(0xffffffffu, ok, 0);
#pragma unroll
    for (int b = 0; b < NSLOT; ++b)
      if (b == sl) loaded[b] = ok;
    ++staged;
    if (++lsp >= sp_end(lu)) {
      ++lu;
      if (lu < u_end) lsp = sp_first(lu);
    }
  };
  for (int k = 0; k < NSLOT - 1; ++k) stage_next();
  if (mode == MODE_CROSS) pdl_wait();
  int qi = -1, qh = -1, m = 0;
  uint32_t qf[4][4];
  bool stop = false;
  for (int u = u_beg; u < u_end && !stop; ++u) {
    const int i = u / (heads * ng), head = (u / ng) % heads, grp = u % ng;
    float RM0 = -INFINITY, RL0 = 0.f, RM1 = -INFINITY, RL1 = 0.f, RA0[16], RA1[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) RA0[k] = RA1[k] = 0.f;
    for (int sp = sp_first(u); sp < sp_end(u); ++sp, ++m) {
      stage_next();                 // walk chunk m + NSLOT - 1 into the slot chunk m - 1 used
      const int cur = m % NSLOT;
      bool have = false;
      uint32_t use = 0u;
#pragma unroll
      for (int b = 0; b < NSLOT; ++b)
        if (b == cur) { have = loaded[b]; use = uses[b]; }
      int k_lo, nk, Lr, nrow;
      unit_range<MODE>(a, i, sp, k_lo, nk, Lr, nrow);
      if (have && (i != qi || head != qh)) {      // query fragments while the chunk lands
        attn_q_frags(reinterpret_cast<const bf16*>(a.Q), a.d, i * H, H, head * WS_DH, qf);
        qi = i;
        qh = head;
      }
      if (have) {
        const bool ok = mbar_wait(&bar[w][cur], use & 1u);
        if (!ok) {               // every slot's copy is waited for (bounded) below
          if (lane == 0) atomicOr(a.status, WS_ST_TIMEOUT);
          stop = true;
          break;
        }
        uint8_t* Ks = slots + cur * CHUNK_BYTES;
        uint8_t* Vs = Ks + CHUNK_BYTES / 2;
        for (int idx = nk * 8 + lane; idx < WS_XCHUNK * 8; idx += 32)   // finite values beyond the keys
          *reinterpret_cast<uint4*>(Vs + idx * 16) = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
        auto vis = [&](int j) -> uint64_t {
          if (j >= H) return 0ull;
          if (mode == MODE_CROSS) return prefix_mask(nk);
          if (j >= nrow) return 0ull;
          return self_key_mask(k_lo, nk, Lr, tree_anc(a.tree, j));
        };
        float m0, l0, m1, l1, acc[8][4];
        // a full chunk that every valid row sees whole (acoustic frames, or
        // cache rows before the block): each mask is all ones or empty
        if (nk == WS_XCHUNK && (mode == MODE_CROSS || k_lo + WS_XCHUNK <= Lr))
          attn_chunk_regs<true, true, true>(Ks, Vs, qf, vis(g), vis(g + 8), m0, l0, m1, l1, acc);
        else
          attn_chunk_regs<true>(Ks, Vs, qf, vis(g), vis(g + 8), m0, l0, m1, l1, acc);
        float a0[16], a1[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          a0[2 * j] = acc[j][0]; a0[2 * j + 1] = acc[j][1];
          a1[2 * j] = acc[j][2]; a1[2 * j + 1] = acc[j][3];
        }
        attn_merge<16>(RM0, RL0, RA0, m0, l0, a0);
        attn_merge<16>(RM1, RL1, RA1, m1, l1, a1);
      }
      __syncwarp();                 // the slot is free for the walk chunk m + NSLOT
#pragma unroll
      for (int b = 0; b < NSLOT; ++b)
        if (b == cur) {
          if (loaded[b]) ++uses[b];
          loaded[b] = false;
        }
    }
    if (stop) break;
    // the group's partial of rows g and g + 8
    auto part = [&](int j) { return a.part + ((((size_t)i * H + j) * heads + head) * ng + grp) * PART; };
    if (g < H) {
      float* p = part(g);
      if (c == 0) { p[0] = RM0; p[1] = RL0; }
#pragma unroll
      for (int j = 0; j < 8; ++j) *reinterpret_cast<float2*>(p + 2 + 8 * j + 2 * c) = make_float2(RA0[2 * j], RA0[2 * j + 1]);
    }
    if (g + 8 < H) {
      float* p = part(g + 8);
      if (c == 0) { p[0] = RM1; p[1] = RL1; }
#pragma unroll
      for (int j = 0; j < 8; ++j) *reinterpret_cast<float2*>(p + 2 + 8 * j + 2 * c) = make_float2(RA1[2 * j], RA1[2 * j + 1]);
    }
  }
  // copies still requested (an early stop) land before exit (bounded)
#pragma unroll
  for (int b = 0; b < NSLOT; ++b)
    if (loaded[b] && lane == 0 && !mbar_wait(&bar[w][b], uses[b] & 1u)) atomicOr(a.status, WS_ST_TIMEOUT);
  __syncwarp();
}

// One warp per (request, row, head): fold the row's group partials in order.
__global__ void __launch_bounds__(512) attn_fold_kernel(AttnArgs a) {
  pdl_wait();
  const int i = blockIdx.x, head = blockIdx.y, j = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads = a.d / WS_DH, ng = (a.n_split + STREAM_GROUP - 1) / STREAM_GROUP;
  pdl_trigger();
  if (j >= a.H) return;
  const float* p = a.part + (((size_t)i * a.H + j) * heads + head) * ng * PART;
  float o0, o1;
  attn_fold_row<false>(p, ng, o0, o1);
  bf16* o = reinterpret_cast<bf16*>(a.O) + ((size_t)i * a.H + j) * a.d + head * WS_DH + 2 * lane;
  o[0] = __float2bfloat16_rn(o0);
  o[1] = __float2bfloat16_rn(o1);
}

// ------------------------------------------------------------------ cluster variant
// One thread-block cluster per (request, head) and one warp per chunk: CTA c
// of a cluster of ceil(n_split / CW) CTAs holds chunks CW * c .. CW * c +
// CW - 1.  Each warp stages its chunk's K and V boxes by TMA (cross-attention
// before the dependency wait, as in the streaming variant) and writes the
// chunk partial (attn_chunk_partial) into its CTA's shared memory.  After a
// cluster barrier the cluster's warps fold the rows (cluster warp g takes
// rows g, g + CW * C, ...) from the partials of every CTA through
// distributed shared memory, in chunk order with the fold kernel's
// arithmetic, and store the attention output: one kernel, no partials in
// global memory, and rows bit-identical to the streaming variant's.
constexpr int CW = 4;                                     // warps (chunks) per CTA
constexpr int CL_MAX = 8;                                 // CTAs per cluster (portable size)
constexpr int CLUSTER_SMEM = CW * CHUNK_BYTES + (CW + 1) * MAXR * PART * 4 + 1024;

template <int MODE>
__global__ void __launch_bounds__(CW * 32) attn_cluster_kernel(const __grid_constant__ CUtensorMap tmKV, AttnArgs a,
                                                                const bf16* kv_base) {
  namespace cg = cooperative_groups;
  extern __shared__ uint8_t dsm_c[];
  __shared__ __align__(8) uint64_t bar[CW];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_c) + 1023) & ~uintptr_t(1023));
  float* parts = reinterpret_cast<float*>(base + CW * CHUNK_BYTES);     // [CW][MAXR][PART]
  cg::cluster_group cl = cg::this_cluster();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = (int)gridDim.x, rank = (int)blockIdx.x;                 // the cluster spans grid.x
  const int head = blockIdx.y, i = blockIdx.z;
  const int heads = a.d / WS_DH, H = a.H, ns = a.n_split;
  const int sp = rank * CW + w;                                        // this warp's chunk
  const int mode = MODE >= 0 ? MODE : a.mode;
  uint8_t* Ks = base + w * CHUNK_BYTES;
  uint8_t* Vs = Ks + CHUNK_BYTES / 2;
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[w])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  pdl_trigger();
  // cross-attention K/V were written before this library call began (see
  // the streaming variant); self-attention reads rows this call wrote
  if (mode == MODE_SELF) pdl_wait();
  bool loaded = false;
  if (lane == 0 && sp < ns) loaded = stage_unit<MODE>(a, &tmKV, kv_base, (i * heads + head) * ns + sp, Ks, &bar[w]);
  loaded = __shfl_sync(0xffffffffu, loaded, 0);
  if (mode == MODE_CROSS) pdl_wait();
  auto part = [&](int j) { return parts + (w * MAXR + j) * PART; };
  bool landed = !loaded;
  if (sp < ns) {
    if (loaded) {
      uint32_t qf[4][4];
      attn_q_frags(reinterpret_cast<const bf16*>(a.Q), a.d, i * H, H, head * WS_DH, qf);   // while the chunk lands
      landed = mbar_wait(&bar[w], 0);
      if (!landed && lane == 0) atomicOr(a.status, WS_ST_TIMEOUT);
      if (landed) {
        int k_lo, nk, Lr, nrow;
        unit_range<MODE>(a, i, sp, k_lo, nk, Lr, nrow);
        for (int idx = nk * 8 + lane; idx < WS_XCHUNK * 8; idx += 32)   // finite values beyond the keys
          *reinterpret_cast<uint4*>(Vs + idx * 16) = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
        auto vis = [&](int j) -> uint64_t {
          if (j >= H) return 0ull;
          if (mode == MODE_CROSS) return prefix_mask(nk);
          if (j >= nrow) return 0ull;
          return self_key_mask(k_lo, nk, Lr, tree_anc(a.tree, j));
        };
        attn_chunk_partial<true>(Ks, Vs, qf, vis(lane >> 2), vis((lane >> 2) + 8), H, part);
      }
    }
    if (!loaded || !landed) {       // no keys here (or the copy timed out): an empty partial
      for (int j = 0; j < H; ++j) {
        float* p = part(j);
        if (lane == 0) { p[0] = -INFINITY; p[1] = 0.f; }
        p[2 + 2 * lane] = 0.f;
        p[3 + 2 * lane] = 0.f;
      }
    }
  }
  // This CTA's four chunks are one group (CW == ATTN_GROUP): merge their
  // partials row by row in chunk order (attn_merge, as the streaming variant
  // does in registers), then fold the cluster's groups through DSMEM with
  // the fold kernel's arithmetic.
  static_assert(CW == ATTN_GROUP, "a CTA's chunks form one partial group");
  __syncthreads();                  // the CTA's chunk partials are written
  float* gparts = parts + CW * MAXR * PART;                       // [MAXR][PART] group partials
  for (int j = w; j < H; j += CW) {
    float GM = -INFINITY, GL = 0.f, GA[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < CW; ++k) {
      if (rank * CW + k >= ns) break;
      const float* p = parts + (k * MAXR + j) * PART;
      const float2 av = *reinterpret_cast<const float2*>(p + 2 + 2 * lane);
      const float aa[2] = {av.x, av.y};
      attn_merge<2>(GM, GL, GA, p[0], p[1], aa);
    }
    float* q = gparts + j * PART;
    if (lane == 0) { q[0] = GM; q[1] = GL; }
    q[2 + 2 * lane] = GA[0];
    q[3 + 2 * lane] = GA[1];
  }
  cl.sync();                        // every group partial of the cluster is written
  for (int j = rank * CW + w; j < H; j += C * CW) {
    float o0, o1;
    attn_fold_row_of<false>([&](int g) { return cl.map_shared_rank(gparts, g) + j * PART; }, C, o0, o1);
    bf16* o = reinterpret_cast<bf16*>(a.O) + ((size_t)i * H + j) * a.d + head * WS_DH + 2 * lane;
    o[0] = __float2bfloat16_rn(o0);
    o[1] = __float2bfloat16_rn(o1);
  }
  cl.sync();                        // peers have read this CTA's partials
  // a copy whose wait timed out lands before exit (bounded)
  if (loaded && !landed && lane == 0 && !mbar_wait(&bar[w], 0)) atomicOr(a.status, WS_ST_TIMEOUT);
  __syncwarp();
}

int g_attn_sms = 0;

// Requests per call up to which the cluster variant runs (one cluster per
// (request, head)); larger calls stream.
constexpr int CLUSTER_MAX_REQ = 4;

template <int MODE>
cudaError_t launch_cluster(const AttnArgs& a, int n, int heads, const CUtensorMap& map, const void* kv_base,
                           cudaStream_t s, bool pdl) {
  const int C = (a.n_split + CW - 1) / CW;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, heads, n);
  cfg.blockDim = dim3(CW * 32);
  cfg.dynamicSmemBytes = CLUSTER_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (pdl) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  at[na].id = cudaLaunchAttributeClusterDimension;
  at[na].val.clusterDim.x = C;
  at[na].val.clusterDim.y = 1;
  at[na].val.clusterDim.z = 1;
  ++na;
  cfg.attrs = at;
  cfg.numAttrs = na;
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<-1>, map, a, reinterpret_cast<const bf16*>(kv_base));
}


template <int MODE>
cudaError_t launch_stream(const AttnArgs& a, int n, int heads, const CUtensorMap& map, const void* kv_base,
                          cudaStream_t s, bool pdl) {
  const int total = n * heads * ((a.n_split + STREAM_GROUP - 1) / STREAM_GROUP);
  const int cap = g_attn_sms > 0 ? g_attn_sms : 148;             // one CTA per SM
  const int ctas = (total + SW - 1) / SW;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas < cap ? ctas : cap);
  cfg.blockDim = dim3(SW * 32);
  cfg.dynamicSmemBytes = STREAM_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  ws_count_launches(1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_stream_kernel<MODE>, map, a, reinterpret_cast<const bf16*>(kv_base));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t f = {};
  f.gridDim = dim3(n, heads);
  f.blockDim = dim3(32 * a.H);
  f.stream = s;
  f.attrs = at;
  f.numAttrs = pdl ? 1 : 0;
  ws_count_launches(1);
  return cudaLaunchKernelEx(&f, attn_fold_kernel, a);
}

template <int MODE>
cudaError_t launch_chunks(const AttnArgs& a, int n, int heads, const CUtensorMap& map, const void* kv_base,
                          cudaStream_t s, bool pdl) {
  if (n <= CLUSTER_MAX_REQ && a.n_split <= CW * CL_MAX && a.H <= MAXR)
    return launch_cluster<MODE>(a, n, heads, map, kv_base, s, pdl);
  return launch_stream<MODE>(a, n, heads, map, kv_base, s, pdl);
}

template <typename T>
constexpr size_t attn_smem() {
  return 2 * SPLIT * WS_DH * sizeof(T) + SPLIT * (WS_DH + 1) * 4 + SPLIT * WS_DH * 4 + MAXR * WS_DH * 4 +
         NW * 32 * 4;
}

template <typename T, int MODE>
cudaError_t launch_mode(const AttnArgs& a, int n, int heads, cudaStream_t s, bool pdl) {
  static bool attr = false;
  constexpr size_t smem = attn_smem<T>();
  if (!attr) {
    cudaError_t r = cudaFuncSetAttribute(attn_split_kernel<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (r != cudaSuccess) return r;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n, heads, a.n_split);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, attn_split_kernel<T, MODE>, a);
}

}  // namespace

template <typename T>
cudaError_t attn_init_attributes() {
  cudaError_t r = cudaSuccess;
  constexpr int smem = (int)attn_smem<T>();
  if (r == cudaSuccess) r = cudaFuncSetAttribute(attn_split_kernel<T, MODE_SELF>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (r == cudaSuccess) r = cudaFuncSetAttribute(attn_split_kernel<T, MODE_CROSS>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (r == cudaSuccess) r = cudaFuncSetAttribute(attn_split_kernel<T, MODE_DRAFT>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (r == cudaSuccess) r = cudaFuncSetAttribute(attn_stream_kernel<MODE_SELF>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, STREAM_SMEM);
  if (r == cudaSuccess) r = cudaFuncSetAttribute(attn_stream_kernel<MODE_CROSS>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, STREAM_SMEM);
  if (r == cudaSuccess) r = cudaFuncSetAttribute(attn_cluster_kernel<-1>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, CLUSTER_SMEM);
  if (r == cudaSuccess) {
    int dev = 0;
    r = cudaGetDevice(&dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&g_attn_sms, cudaDevAttrMultiProcessorCount, dev);
  }
  return r;
}

template <typename T>
cudaError_t launch_self_attn(int n, int H, const RowMap& rm, const TreeMask& tree, const T* Q, const KVPool& kv, T* O,
                             int n_heads, const AttnScratch& sc, cudaStream_t s, bool pdl) {
  if (H > MAXR) return cudaErrorInvalidValue;
  AttnArgs a = {};
  a.tree = tree;
  a.mode = MODE_SELF;
  a.H = H; a.d = n_heads * WS_DH; a.max_pos = rm.max_pos;
  a.n_split = (rm.max_pos + SPLIT - 1) / SPLIT;
  a.req_ids = rm.req_ids; a.L = rm.L; a.block_len = rm.block_len;
  a.Q = Q; a.kv = kv; a.part = sc.part; a.counters = sc.counters; a.O = O; a.status = sc.status;
  a.n_req = n;
  if (sizeof(T) == 2 && sc.kv_map)
    return launch_chunks<MODE_SELF>(a, n, n_heads, *reinterpret_cast<const CUtensorMap*>(sc.kv_map), sc.kv_base, s,
                                    pdl);
  return launch_mode<T, MODE_SELF>(a, n, n_heads, s, pdl);
}

template <typename T>
cudaError_t launch_cross_attn(int n, int H, const int32_t* req_ids, const int32_t* Fv, const T* Q, const XKV& x,
                              int layer, T* O, int n_heads, int max_frames_seen, const AttnScratch& sc,
                              cudaStream_t s, bool pdl) {
  if (H > MAXR) return cudaErrorInvalidValue;
  AttnArgs a = {};
  a.mode = MODE_CROSS;
  a.H = H; a.d = n_heads * WS_DH;
  a.n_split = max(1, (max_frames_seen + SPLIT - 1) / SPLIT);
  a.req_ids = req_ids; a.Fv = Fv; a.Q = Q; a.x = x; a.xlayer = layer;
  a.part = sc.part; a.counters = sc.counters; a.O = O; a.status = sc.status;
  a.n_req = n;
  if (sizeof(T) == 2 && sc.xkv_map)
    return launch_chunks<MODE_CROSS>(a, n, n_heads, *reinterpret_cast<const CUtensorMap*>(sc.xkv_map), x.base, s,
                                     pdl);
  return launch_mode<T, MODE_CROSS>(a, n, n_heads, s, pdl);
}

template <typename T>
cudaError_t launch_draft_attn(int n, int K1, const int32_t* req_ids, const int32_t* L, const T* Q, const T* Kb,
                              const T* Vb, const KVPool& hkv, T* O, int n_heads, int max_pos,
                              const AttnScratch& sc, cudaStream_t s, bool pdl) {
  if (K1 > MAXR) return cudaErrorInvalidValue;
  AttnArgs a = {};
  a.mode = MODE_DRAFT;
  a.H = K1; a.d = n_heads * WS_DH; a.max_pos = max_pos;
  a.n_split = (max_pos + SPLIT - 1) / SPLIT + 1;
  a.req_ids = req_ids; a.L = L; a.Q = Q; a.kv = hkv; a.Kb = Kb; a.Vb = Vb;
  a.part = sc.part; a.counters = sc.counters; a.O = O; a.status = sc.status;
  return launch_mode<T, MODE_DRAFT>(a, n, n_heads, s, pdl);
}

#define INST(T)                                                                                                  \
  template cudaError_t attn_init_attributes<T>();                                                               \
  template cudaError_t launch_self_attn<T>(int, int, const RowMap&, const TreeMask&, const T*, const KVPool&, T*, int,            \
                                           const AttnScratch&, cudaStream_t, bool);                              \
  template cudaError_t launch_cross_attn<T>(int, int, const int32_t*, const int32_t*, const T*, const XKV&, int, \
                                            T*, int, int, const AttnScratch&, cudaStream_t, bool);               \
  template cudaError_t launch_draft_attn<T>(int, int, const int32_t*, const int32_t*, const T*, const T*,        \
                                            const T*, const KVPool&, T*, int, int, const AttnScratch&,           \
                                            cudaStream_t, bool);
INST(float)
INST(bf16)
