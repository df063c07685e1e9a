// Attention arithmetic shared by the per-op attention kernel and the
// persistent block-verification kernel, so both produce bit-identical rows:
// the online-softmax update of one query row over up to 32 keys, and the
// fold of per-split partials (max, sum, 64 weighted values) in split order.
#pragma once
#include "ws_internal.cuh"

constexpr int WS_ATTN_PART = WS_DH + 2;    // floats per split partial

struct RowState { float m, l, a0, a1; };

// Keys 0 .. n-1 of a chunk of 64.
__device__ __forceinline__ uint64_t prefix_mask(int n) {
  return n >= 64 ? ~0ull : (n <= 0 ? 0ull : ((1ull << n) - 1ull));
}
// Self-attention keys of the chunk [k_lo, k_lo + nk) that a block row sees:
// every cache key before the block start L, and of the block's own slots L,
// L + 1, ... those whose bit is set in anc (the row's ancestors in the
// candidate tree; rows 0..j for a linear block).
__device__ __forceinline__ uint64_t self_key_mask(int k_lo, int nk, int L, uint32_t anc) {
  const int sh = L - k_lo;
  uint64_t m = prefix_mask(sh);
  if (sh >= 0 && sh < 64) m |= (uint64_t)anc << sh;
  else if (sh < 0 && sh > -32) m |= (uint64_t)(anc >> (-sh));
  return m & prefix_mask(nk);
}

// One sub-tile of up to 32 keys for one row (warp-wide): scores by lane = key,
// online-softmax update, then weighted values with lane = pair of dims.
// Keys whose bit in vmask is clear get no weight; the first key of every
// sub-tile a row visits is visible (the keys before the block start are).
__device__ __forceinline__ void row_subtile(RowState& st, const float* q, const float (*Kt)[WS_DH + 1],
                                            const float (*Vt)[WS_DH], int k0, int nvalid, float* pw,
                                            uint32_t vmask = 0xFFFFFFFFu) {
  const int lane = threadIdx.x & 31;
  float s = -INFINITY;
  if (lane < nvalid && ((vmask >> lane) & 1u)) {
    const float* kr = Kt[k0 + lane];
    float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll
    for (int d = 0; d < WS_DH; d += 4) {
      c0 = fmaf(q[d], kr[d], c0);
      c1 = fmaf(q[d + 1], kr[d + 1], c1);
      c2 = fmaf(q[d + 2], kr[d + 2], c2);
      c3 = fmaf(q[d + 3], kr[d + 3], c3);
    }
    s = ((c0 + c1) + (c2 + c3)) * 0.125f;          // 1/sqrt(64)
  }
  const float mn = fmaxf(st.m, warp_max(s));
  const float p = lane < nvalid ? expf(s - mn) : 0.0f;
  const float corr = expf(st.m - mn);
  st.l = st.l * corr + warp_sum(p);
  pw[lane] = p;
  __syncwarp();
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
  int k = 0;
  for (; k + 1 < nvalid; k += 2) {
    const float2 v = *reinterpret_cast<const float2*>(&Vt[k0 + k][2 * lane]);
    const float2 w = *reinterpret_cast<const float2*>(&Vt[k0 + k + 1][2 * lane]);
    a0 = fmaf(pw[k], v.x, a0); a1 = fmaf(pw[k], v.y, a1);
    b0 = fmaf(pw[k + 1], w.x, b0); b1 = fmaf(pw[k + 1], w.y, b1);
  }
  if (k < nvalid) {
    const float2 v = *reinterpret_cast<const float2*>(&Vt[k0 + k][2 * lane]);
    a0 = fmaf(pw[k], v.x, a0); a1 = fmaf(pw[k], v.y, a1);
  }
  __syncwarp();
  st.a0 = st.a0 * corr + (a0 + b0);
  st.a1 = st.a1 * corr + (a1 + b1);
  st.m = mn;
}

// Fold the partials of one row, splits s = 0 .. n_split-1 in order, split s
// at part_of(s) (m, l, 64 weighted values); lane l returns output dims (2l,
// 2l+1).  GLOBAL: the partials are in global memory, written by other CTAs
// (read from L2); else in this cluster's shared memory (generic loads).  All
// loads of a group of splits are issued before their values are used (one
// round trip per group instead of one per split); the arithmetic and its
// order are those of the sequential fold: M = max_s m_s, then den, n0, n1
// accumulate over s = 0, 1, ... with weights exp(m_s - M), skipping empty
// splits.
// Chunks per partial group: the partials of ATTN_GROUP consecutive 64-key
// chunks of a row are merged in chunk order (attn_merge), and the group
// partials are folded in group order (attn_fold_row_of).  Every bf16
// attention kernel of the batched and one-cluster paths does exactly this,
// so a row's result does not depend on how many requests share the call.
constexpr int ATTN_GROUP = 4;

// Merge one chunk partial (m, l, a[K]) into the running group partial (M, L,
// A[K]); empty chunks (l = 0) are skipped and the first non-empty chunk is
// taken as is.  Explicit FMAs fix the rounding in every kernel.
template <int K>
__device__ __forceinline__ void attn_merge(float& M, float& L, float* A, float m, float l, const float* a) {
  if (!(l > 0.f)) return;
  if (!(L > 0.f)) {
    M = m;
    L = l;
#pragma unroll
    for (int k = 0; k < K; ++k) A[k] = a[k];
    return;
  }
  // the larger of M and m keeps weight exp(0) = 1: one exponential per merge
  const bool up = m > M;
  const float e = expf(up ? M - m : m - M);
  const float cr = up ? e : 1.0f, cn = up ? 1.0f : e;
  L = fmaf(L, cr, __fmul_rn(l, cn));
#pragma unroll
  for (int k = 0; k < K; ++k) A[k] = fmaf(A[k], cr, __fmul_rn(a[k], cn));
  M = up ? m : M;
}

template <bool GLOBAL>
__device__ __forceinline__ float fold_ld(const float* p) { return GLOBAL ? __ldcg(p) : *p; }
template <bool GLOBAL>
__device__ __forceinline__ float2 fold_ld2(const float* p) {
  return GLOBAL ? __ldcg(reinterpret_cast<const float2*>(p)) : *reinterpret_cast<const float2*>(p);
}

template <bool GLOBAL, bool ONE_TRIP = true, class PartOf>
__device__ __forceinline__ void attn_fold_row_of(PartOf part_of, int n_split, float& o0, float& o1) {
  const int lane = threadIdx.x & 31;
  if (ONE_TRIP && n_split <= 32) {
    // every load at once (one round trip): split `lane`'s (m, l) and each
    // split's two output dims of this lane; same arithmetic as below
    const float2 ml = lane < n_split ? fold_ld2<GLOBAL>(part_of(lane)) : make_float2(-INFINITY, 0.f);
    float2 av[32];
#pragma unroll
    for (int u = 0; u < 32; ++u)
      if (u < n_split) av[u] = fold_ld2<GLOBAL>(part_of(u) + 2 + 2 * lane);
    const float M = fmaxf(-INFINITY, warp_max(ml.x));
    float den = 0.f, n0 = 0.f, n1 = 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      if (u >= n_split) break;
      const float l = __shfl_sync(0xffffffffu, ml.y, u);
      const float m = __shfl_sync(0xffffffffu, ml.x, u);
      if (l <= 0.f) continue;
      const float c = expf(m - M);
      den = fmaf(l, c, den);
      n0 = fmaf(av[u].x, c, n0);
      n1 = fmaf(av[u].y, c, n1);
    }
    o0 = den > 0.f ? n0 / den : 0.f;
    o1 = den > 0.f ? n1 / den : 0.f;
    return;
  }
  float M = -INFINITY;
  for (int s0 = 0; s0 < n_split; s0 += 32) {
    const int s = s0 + lane;
    const float m = s < n_split ? fold_ld<GLOBAL>(part_of(s)) : -INFINITY;
    M = fmaxf(M, warp_max(m));
  }
  float den = 0.f, n0 = 0.f, n1 = 0.f;
  for (int s0 = 0; s0 < n_split; s0 += 32) {
    const int sl = s0 + lane;
    float2 ml = make_float2(-INFINITY, 0.f);
    if (sl < n_split) ml = fold_ld2<GLOBAL>(part_of(sl));
    const int nin = min(32, n_split - s0);
    for (int t = 0; t < nin; t += 8) {
      float2 av[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (t + u < nin) av[u] = fold_ld2<GLOBAL>(part_of(s0 + t + u) + 2 + 2 * lane);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (t + u >= nin) break;
        const float l = __shfl_sync(0xffffffffu, ml.y, t + u);
        const float m = __shfl_sync(0xffffffffu, ml.x, t + u);
        if (l <= 0.f) continue;
        const float c = expf(m - M);
        den = fmaf(l, c, den);
        n0 = fmaf(av[u].x, c, n0);
        n1 = fmaf(av[u].y, c, n1);
      }
    }
  }
  o0 = den > 0.f ? n0 / den : 0.f;
  o1 = den > 0.f ? n1 / den : 0.f;
}

// Partials p[s * WS_ATTN_PART] in global memory.  ONE_TRIP = false keeps
// the register footprint small (grouped loads); the result is the same.
template <bool ONE_TRIP = true>
__device__ __forceinline__ void attn_fold_row(const float* p, int n_split, float& o0, float& o1) {
  attn_fold_row_of<true, ONE_TRIP>([p](int s) { return p + (size_t)s * WS_ATTN_PART; }, n_split, o0, o1);
}
