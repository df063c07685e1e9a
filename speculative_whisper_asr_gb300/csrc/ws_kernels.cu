// Element-wise and per-request kernels of the decoding path: embeddings,
// layer norm, argmax bookkeeping, history gather, sampling, acceptance.
#include "ws_internal.cuh"

namespace {

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                            cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

// Block-wide fixed-order reductions (blockDim.x == 256 or 128).
template <int NT>
__device__ float block_sum(float v, float* sh) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t += sh[i];
  return t;
}
template <int NT>
__device__ float block_max(float v, float* sh) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  float t = -INFINITY;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t = fmaxf(t, sh[i]);
  return t;
}

// ------------------------------------------------------------------ embeddings
// Target rows: x = E[token] + P[position] (token + learned position embedding).
// Block row j sits at position L + depth(j) (depth(j) = j for a linear block,
// the tree depth for a candidate tree); its cache slot L + j is checked.
template <typename T>
__global__ void embed_target_kernel(RowMap rm, unsigned long long depth4, const int32_t* block, const T* E,
                                    const T* P, int d, int V, float* x, int32_t* pend_start, int32_t* pend_n,
                                    int32_t* status) {
  pdl_wait();
  const int r = blockIdx.x;
  int slot, j, pos;
  bool valid = row_info(rm, r, slot, j, pos);         // pos: the row's cache slot L + j
  const int i = r / rm.H;
  int tok = block[r];
  bool in_block = j < rm.block_len[i];
  if (in_block && pos >= rm.max_pos && threadIdx.x == 0) atomicOr(status, WS_ST_POS);
  pos -= j - tree_depth(depth4, j);                   // the embedded position L + depth(j) <= L + j
  if (!valid) { tok = 0; pos = min(pos, rm.max_pos - 1); }
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) atomicOr(status, WS_ST_TOKEN);
    tok = 0;
  }
  if (j == 0 && threadIdx.x == 0) {
    pend_start[slot] = rm.L[slot];
    pend_n[slot] = rm.block_len[i];
  }
  pdl_trigger();
  const T* e = E + (size_t)tok * d;
  const T* p = P + (size_t)pos * d;
  for (int n = threadIdx.x; n < d; n += blockDim.x) x[(size_t)r * d + n] = to_f<T>(e[n]) + to_f<T>(p[n]);
}

// Drafter rows: X_t = [Emb(anchor), m, ..., m] (Whisper-Flash Eq. 2); no
// absolute position embedding (positions enter through RoPE).
template <typename T>
__global__ void embed_draft_kernel(int K1, const int32_t* req_ids, const int32_t* block, const T* E, const T* m,
                                   int d, int V, float* x, int32_t* pend_n, int32_t* status) {
  pdl_wait();
  const int r = blockIdx.x, i = r / K1, j = r - i * K1;
  const T* src = m;
  if (j == 0) {
    int tok = block[(size_t)i * K1];
    if (tok < 0 || tok >= V) {
      if (threadIdx.x == 0) atomicOr(status, WS_ST_TOKEN);
      tok = 0;
    }
    src = E + (size_t)tok * d;
    if (threadIdx.x == 0) pend_n[req_ids[i]] = 0;   // history rows are folded in by now
  }
  pdl_trigger();
  for (int n = threadIdx.x; n < d; n += blockDim.x) x[(size_t)r * d + n] = to_f<T>(src[n]);
}

// ------------------------------------------------------------------ layer norm
// y = (x - mean) / sqrt(var + 1e-5) * g + b over each row, fp32 statistics.
// group_skip > 0: output row o reads input row (o / (G-1)) * G + o % (G-1) + 1
// (drops row 0 of every group of G rows: the drafter's anchor row).
// One warp per row (ln_row_warp), four rows per CTA; bf16 rows are stored
// four values (8 bytes) at a time.  MAXV: register groups of 128 features
// (d <= 128 * MAXV).
template <typename T, int MAXV>
__global__ void __launch_bounds__(128) layernorm_kernel(int M, int d, const float* x, int ldx, const T* g,
                                                        const T* b, T* y, int ldy, int group_skip) {
  pdl_trigger();
  // gain and bias are weights: bring this lane's groups into L1 before the
  // dependency wait, so the normalisation does not wait on L2 after the
  // reductions
  const int lane = threadIdx.x & 31;
  for (int k = 4 * lane; k < d; k += 128) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(g + k));
    asm volatile("prefetch.global.L1 [%0];" ::"l"(b + k));
  }
  pdl_wait();
  const int o = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (o >= M) return;
  int src = o;
  if (group_skip > 0) {
    int G1 = group_skip - 1;
    src = (o / G1) * group_skip + (o % G1) + 1;
  }
  T* yr = y + (size_t)o * ldy;
  ln_row_warp<false, MAXV>(x + (size_t)src * ldx, d, g, b, sizeof(T) == 2, [&](int k, float a0, float a1, float a2, float a3) {
    if constexpr (sizeof(T) == 2) {
      __nv_bfloat162 h0 = __floats2bfloat162_rn(a0, a1), h1 = __floats2bfloat162_rn(a2, a3);
      uint2 w;
      w.x = *reinterpret_cast<uint32_t*>(&h0);
      w.y = *reinterpret_cast<uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(yr + k) = w;
    } else {
      yr[k] = from_f<T>(a0); yr[k + 1] = from_f<T>(a1); yr[k + 2] = from_f<T>(a2); yr[k + 3] = from_f<T>(a3);
    }
  });
}

// Many rows (the encoder's 1500 per window): gain and bias are staged in
// shared memory once per CTA, and each warp normalises LN_RPW consecutive
// rows two at a time (both rows' loads in one memory round trip), with the
// same per-row arithmetic as layernorm_kernel.
constexpr int LN_RPW = 4;
constexpr int LN_MANY = 4096;     // rows from which a call takes this kernel
template <typename T, int MAXV>
__global__ void __launch_bounds__(128) layernorm_rows_kernel(int M, int d, const float* x, int ldx, const T* g,
                                                             const T* b, T* y, int ldy, int group_skip) {
  __shared__ __align__(16) T gb[2][128 * MAXV];
  pdl_trigger();
  constexpr int PER = 8 / sizeof(T);             // elements per 8-byte copy
  for (int i = threadIdx.x * PER; i < d; i += 128 * PER) {
    *reinterpret_cast<uint2*>(&gb[0][i]) = *reinterpret_cast<const uint2*>(g + i);
    *reinterpret_cast<uint2*>(&gb[1][i]) = *reinterpret_cast<const uint2*>(b + i);
  }
  __syncthreads();
  pdl_wait();
  const int o0 = (blockIdx.x * 4 + (threadIdx.x >> 5)) * LN_RPW;
  for (int j = 0; j < LN_RPW; j += 2) {
    const int oa = o0 + j;
    if (oa >= M) break;
    const int nr = min(2, M - oa);
    const float* xs[2];
    T* ys[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int o = oa + (r < nr ? r : 0);
      int src = o;
      if (group_skip > 0) {
        const int G1 = group_skip - 1;
        src = (o / G1) * group_skip + (o % G1) + 1;
      }
      xs[r] = x + (size_t)src * ldx;
      ys[r] = y + (size_t)o * ldy;
    }
    ln_rows_warp<false, 2, MAXV>(xs, nr, d, gb[0], gb[1], sizeof(T) == 2,
                                 [&](int r, int k, float a0, float a1, float a2, float a3) {
      T* yr = ys[r];
      if constexpr (sizeof(T) == 2) {
        __nv_bfloat162 h0 = __floats2bfloat162_rn(a0, a1), h1 = __floats2bfloat162_rn(a2, a3);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t*>(&h0);
        w.y = *reinterpret_cast<uint32_t*>(&h1);
        *reinterpret_cast<uint2*>(yr + k) = w;
      } else {
        yr[k] = from_f<T>(a0); yr[k + 1] = from_f<T>(a1); yr[k + 2] = from_f<T>(a2); yr[k + 3] = from_f<T>(a3);
      }
    });
  }
}

// ------------------------------------------------------------------ argmax
__global__ void argmax_init_kernel(int M, unsigned long long* keys) {
  pdl_wait();
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < M) keys[i] = 0ull;
  pdl_trigger();
}

// keys [n*H] -> out[i*stride + col0 + j]; rows j >= block_len[i] get -1.
__global__ void argmax_finalize_kernel(int n, int H, const int32_t* block_len, const unsigned long long* keys,
                                       int32_t* out, int stride, int col0) {
  pdl_wait();
  int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < n * H) {
    int i = r / H, j = r - i * H;
    bool valid = block_len ? (j < block_len[i]) : true;
    out[(size_t)i * stride + col0 + j] = valid ? argmax_key_id(keys[r]) : -1;
  }
  pdl_trigger();
}

// ------------------------------------------------------------------ history gather
// feat[i*Hp + j] = concat_h resid_h(slot, j) for pending rows (else zeros);
// the concatenated residual streams are the fusion projection's input.
template <typename T>
__global__ void hist_gather_kernel(int Hp, const int32_t* req_ids, const int32_t* pend_n, const float* hist,
                                   int max_block, int n_hist, int d, T* feat) {
  pdl_wait();
  const int r = blockIdx.x, i = r / Hp, j = r - i * Hp;
  const int slot = req_ids[i];
  const bool valid = j < pend_n[slot];
  const int w = n_hist * d;
  const float* src = hist + ((size_t)slot * max_block + j) * w;
  pdl_trigger();
  for (int c = threadIdx.x; c < w; c += blockDim.x) feat[(size_t)r * w + c] = from_f<T>(valid ? src[c] : 0.0f);
}

// ------------------------------------------------------------------ RoPE table
// tab[pos][i] = (cos, sin)(fp32(pos * theta_i)), theta_i = fp32(10000^(-2i/64)):
// base 10,000 and FP32 phases (Whisper-Flash Appendix A.2).  The cos/sin of the
// fp32 phase are evaluated in double and rounded once.
__global__ void rope_table_kernel(float* tab, int max_pos) {
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= max_pos * (WS_DH / 2)) return;
  int pos = idx / (WS_DH / 2), i = idx % (WS_DH / 2);
  float theta = (float)pow(10000.0, -2.0 * (double)i / (double)WS_DH);
  float ang = (float)pos * theta;
  tab[idx * 2 + 0] = (float)cos((double)ang);
  tab[idx * 2 + 1] = (float)sin((double)ang);
}

// ------------------------------------------------------------------ request state
__global__ void set_frames_kernel(int n, const int32_t* req_ids, const int32_t* cu, const int32_t* valid,
                                  int max_frames, int32_t* Fc, int32_t* Fv, int32_t* status) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int F = cu[i + 1] - cu[i];
  int v = valid ? valid[i] : F;
  if (F < 0 || F > max_frames || v < 0 || v > F) {
    atomicOr(status, WS_ST_FRAMES);
    F = max(0, min(F, max_frames));
    v = max(0, min(v, F));
  }
  Fc[req_ids[i]] = F;
  Fv[req_ids[i]] = v;
}

__global__ void reset_kernel(int n, const int32_t* req_ids, int32_t* L, int32_t* pend_n, int32_t* xcenter) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) { L[req_ids[i]] = 0; pend_n[req_ids[i]] = 0; xcenter[req_ids[i]] = -1; }
}

__global__ void get_lengths_kernel(int n, const int32_t* req_ids, const int32_t* L, int32_t* out) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = L[req_ids[i]];
}

// ------------------------------------------------------------------ sampling helpers
constexpr int SNT = 256;   // threads of the sampling / acceptance CTAs

__device__ __forceinline__ bool suppressed(const uint32_t* sup, int v) {
  return sup && ((sup[v >> 5] >> (v & 31)) & 1u);
}
// Scaled logit z/T (suppressed ids -> -inf).
__device__ __forceinline__ float scaled(const float* z, int v, float T, const uint32_t* sup) {
  return suppressed(sup, v) ? -INFINITY : z[v] / T;
}
// The same for an already loaded logit value zv of id v.
__device__ __forceinline__ float scaled_val(float zv, int v, float T, const uint32_t* sup) {
  return suppressed(sup, v) ? -INFINITY : zv / T;
}

struct RowStat { float m, S; };
// max and sum of exp(z/T - max) over a row (FP32).  Each thread takes ids
// tid, tid + 256, ... with sixteen loads in flight (the row streams from
// HBM at microseconds of latency): four partial maxima / sums combined in a
// fixed order, then the block reduces in a fixed order.  The maximum is
// taken over the raw logits and divided once: a correctly rounded division
// by T > 0 is monotone, so max(z) / T equals max(z / T) exactly.
constexpr int RS_DEPTH = 16;
__device__ RowStat row_stat(const float* z, int V, float T, const uint32_t* sup, float* sh) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  int v = threadIdx.x;
  for (; v + (RS_DEPTH - 1) * SNT < V; v += RS_DEPTH * SNT) {
    float zz[RS_DEPTH];
#pragma unroll
    for (int q = 0; q < RS_DEPTH; ++q) zz[q] = __ldg(z + v + q * SNT);      // all loads first
#pragma unroll
    for (int q = 0; q < RS_DEPTH; ++q) m4[q & 3] = fmaxf(m4[q & 3], suppressed(sup, v + q * SNT) ? -INFINITY : zz[q]);
  }
  for (; v < V; v += SNT) m4[0] = fmaxf(m4[0], suppressed(sup, v) ? -INFINITY : z[v]);
  const float m = block_max<SNT>(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])), sh) / T;
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  v = threadIdx.x;
  for (; v + (RS_DEPTH - 1) * SNT < V; v += RS_DEPTH * SNT) {
    float zz[RS_DEPTH];
#pragma unroll
    for (int q = 0; q < RS_DEPTH; ++q) zz[q] = __ldg(z + v + q * SNT);
#pragma unroll
    for (int q = 0; q < RS_DEPTH; ++q) s4[q & 3] += expf(scaled_val(zz[q], v + q * SNT, T, sup) - m);
  }
  for (; v < V; v += SNT) s4[0] += expf(scaled(z, v, T, sup) - m);
  const float s = block_sum<SNT>((s4[0] + s4[1]) + (s4[2] + s4[3]), sh);
  RowStat r; r.m = m; r.S = s;
  return r;
}

__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Float-float sums: TwoSum (Knuth) keeps the rounding error of every FP32
// addition, so a 32-value sum is exact to ~2^-48 relative without FP64
// arithmetic (which runs far slower than FP32 on this part).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
__device__ __forceinline__ void warp_sum_ff(float& hi, float& lo) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o), l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    float sum, err;
    two_sum(hi, h2, sum, err);
    hi = sum;
    lo = (lo + l2) + err;
  }
}

// Inverse CDF over non-negative weights w(v), v = 0..V-1 in ascending id
// order: the smallest v whose running sum exceeds u * sum(w).  Warp k owns
// the contiguous ids [k * seg, (k + 1) * seg), seg a multiple of 256: 256-id
// super-rows of eight coalesced 32-id rows.  Each lane sums its eight ids of
// a super-row with TwoSum and the warp combines the lanes (float-float), so
// every super-row's sum is exact to ~2^-48 and is kept (as FP64) in shared
// memory; sixteen ids per lane are in flight.  Segment sums are prefixed in
// warp order; the warp whose segment holds the target finds the super-row
// from the sums (one per lane, FP64 scan), reloads its eight rows to find the
// row, then the id inside the row with an inclusive float-float warp scan.
constexpr int CDF_SUPER = 8;        // 32-id rows per super-row
constexpr int CDF_SROWS = 32;       // super-rows per warp: V <= 8 * 32 * 256 = 65,536
// rsum_base: the caller's shared scratch of (SNT / 32) * CDF_SROWS doubles (one per kernel).
template <class WF>
__device__ int block_inverse_cdf(WF w, int V, float u, double* rsum_base) {
  // The weights are FP32 probabilities; their running sums are kept exact so
  // that the drawn id depends on the weights, not on the summation order.
  constexpr int NWARP = SNT / 32, SR = CDF_SUPER * 32;
  __shared__ int found;
  __shared__ double shd[NWARP + 1];
  double (*rsum)[CDF_SROWS] = reinterpret_cast<double (*)[CDF_SROWS]>(rsum_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = ((V + NWARP - 1) / NWARP + SR - 1) / SR * SR;
  const int nsr = min(seg / SR, CDF_SROWS);
  const int lo = warp * seg, hi = min(V, lo + seg);
  for (int s0 = 0; s0 < nsr; s0 += 2) {
    float wv[2][CDF_SUPER];
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int q = 0; q < CDF_SUPER; ++q) {
        const int v = lo + SR * (s0 + p) + 32 * q + lane;
        wv[p][q] = (s0 + p < nsr && v < hi) ? w(v) : 0.0f;
      }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      float h = 0.0f, l = 0.0f;
#pragma unroll
      for (int q = 0; q < CDF_SUPER; ++q) {
        float sm, er;
        two_sum(h, wv[p][q], sm, er);
        h = sm;
        l += er;
      }
      warp_sum_ff(h, l);
      if (lane == 0 && s0 + p < nsr) rsum[warp][s0 + p] = (double)h + (double)l;
    }
  }
  __syncwarp();
  // lane l owns super-row l: its sum in FP64, then the segment's
  const double own = lane < nsr ? rsum[warp][lane] : 0.0;
  double incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const double s = __shfl_sync(0xffffffffu, incl, 31);
  __syncthreads();
  if (lane == 0) shd[warp] = s;
  if (threadIdx.x == 0) found = -1;
  __syncthreads();
  if (threadIdx.x == 0) {
    double run = 0.0;
    for (int t = 0; t < NWARP; ++t) { double c = shd[t]; shd[t] = run; run += c; }
    shd[NWARP] = run;
  }
  __syncthreads();
  const double total = shd[NWARP];
  const double target = (double)u * total;
  const double pre = shd[warp];
  const double nxt = warp + 1 < NWARP ? shd[warp + 1] : total;
  if (s > 0.0 && pre <= target && target < nxt) {
    double ex = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) ex = 0.0;
    const unsigned hits = __ballot_sync(0xffffffffu, own > 0.0 && pre + incl > target);
    int tok = -1;
    if (hits) {
      const int sr = __ffs(hits) - 1;
      double before = pre + __shfl_sync(0xffffffffu, ex, sr);
      const int base = lo + SR * sr;
      float wv[CDF_SUPER];
#pragma unroll
      for (int q = 0; q < CDF_SUPER; ++q) {
        const int v = base + 32 * q + lane;
        wv[q] = v < hi ? w(v) : 0.0f;
      }
      // the super-row's rows in order (exact sums, the same in every lane);
      // if rounding leaves the target past them: the last row with weight
      int row = -1, lrow = -1;
      float rw = 0.0f, lrw = 0.0f;
#pragma unroll
      for (int q = 0; q < CDF_SUPER; ++q) {
        float h = wv[q], l = 0.0f;
        warp_sum_ff(h, l);
        const double c = (double)h + (double)l;
        if (c > 0.0) { lrow = q; lrw = wv[q]; }
        if (row < 0) {
          if (c > 0.0 && before + c > target) { row = q; rw = wv[q]; }
          else before += c;
        }
      }
      const bool past = row < 0;
      if (past) { row = lrow; rw = lrw; }
      if (row >= 0) {
        const int v = base + 32 * row + lane;
        float xh = rw, xl = 0.0f;              // inclusive float-float scan of the row
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float yh = __shfl_up_sync(0xffffffffu, xh, o), yl = __shfl_up_sync(0xffffffffu, xl, o);
          if (lane >= o) {
            float sum, err;
            two_sum(xh, yh, sum, err);
            xh = sum;
            xl = (xl + yl) + err;
          }
        }
        const unsigned hit =
            __ballot_sync(0xffffffffu, !past && v < hi && before + ((double)xh + (double)xl) > target);
        const unsigned posw = __ballot_sync(0xffffffffu, rw > 0.0f);
        tok = hit ? base + 32 * row + __ffs(hit) - 1 : (posw ? base + 32 * row + 31 - __clz(posw) : -1);
      }
    }
    if (tok < 0) {   // rounding left the target past the rows: last id with weight in the segment
      for (int k = nsr - 1; k >= 0 && tok < 0; --k) {
        if (!(rsum[warp][k] > 0.0)) continue;
        for (int q = CDF_SUPER - 1; q >= 0 && tok < 0; --q) {
          const int v = lo + SR * k + 32 * q + lane;
          const unsigned posw = __ballot_sync(0xffffffffu, v < hi && w(v) > 0.0f);
          if (posw) tok = lo + SR * k + 32 * q + 31 - __clz(posw);
        }
      }
    }
    if (lane == 0 && tok >= 0) atomicMax(&found, tok);
  }
  __syncthreads();
  if (found < 0) {   // rounding pushed the target past the end: last id with weight
    if (threadIdx.x == 0) {
      for (int vb = V - 1; vb >= 0; --vb) if (w(vb) > 0.0f) { found = vb; break; }
      if (found < 0) found = 0;
    }
    __syncthreads();
  }
  int res = found;
  __syncthreads();
  return res;
}

// One sampled token per (request, row): softmax(z / T) via inverse CDF with
// Philox counter (slot, round, row + 1, 0) — the drafter's sampler.
__global__ void __launch_bounds__(SNT) sample_rows_kernel(int rows, const int32_t* req_ids, const float* logits,
                                                          long long row_stride, int V, float T, uint64_t seed,
                                                          uint64_t rnd, const uint32_t* sup, int32_t* out,
                                                          int out_stride, int out_col0) {
  __shared__ double cdf_scratch[(SNT / 32) * CDF_SROWS];
  __shared__ float sh[SNT + 8];
  pdl_wait();
  const int i = blockIdx.x / rows, r = blockIdx.x - i * rows;
  const int slot = req_ids[i];
  const float* z = logits + ((long long)i * rows + r) * row_stride;
  RowStat st = row_stat(z, V, T, sup, sh);
  const float u = ws_uniform(seed, (uint32_t)slot, rnd, (uint32_t)(r + 1), 0u);
  int tok = block_inverse_cdf([&](int v) { return expf(scaled(z, v, T, sup) - st.m) / st.S; }, V, u, cdf_scratch);
  pdl_trigger();
  if (threadIdx.x == 0) out[(size_t)i * out_stride + out_col0 + r] = tok;
}

// (max, sum exp) of softmax(z / T) for every row of a [n][rows] block of
// logits rows (row_stat, one CTA per row): the statistics the acceptance
// kernel needs for p and q, computed in parallel instead of per request.
__global__ void __launch_bounds__(SNT) row_stats_kernel(const float* logits, int rows, int V, float T,
                                                        const uint32_t* sup, float2* out) {
  __shared__ float sh[SNT + 8];
  pdl_wait();
  const RowStat st = row_stat(logits + (long long)blockIdx.x * V, V, T, sup, sh);
  pdl_trigger();
  if (threadIdx.x == 0) out[blockIdx.x] = make_float2(st.m, st.S);
}

// ------------------------------------------------------------------ limited proposals
// Confidence of drafted token j of request i: its probability under the
// drafter's softmax at temperature T (1 for greedy proposals), FP32, with the
// shared token suppression.  One CTA per (j, i).
__global__ void __launch_bounds__(SNT) draft_conf_kernel(const int32_t* block, int stride, const float* q, int K,
                                                         int V, float T, const uint32_t* sup, float* conf) {
  __shared__ float sh[SNT + 8];
  pdl_wait();
  const int j = blockIdx.x, i = blockIdx.y;
  const float* z = q + ((long long)i * K + j) * V;
  const RowStat st = row_stat(z, V, T, sup, sh);
  pdl_trigger();
  if (threadIdx.x == 0) {
    const int y = block[(size_t)i * stride + 1 + j];
    conf[(size_t)i * K + j] = (y >= 0 && y < V) ? expf(scaled(z, y, T, sup) - st.m) / st.S : 0.0f;
  }
}

// Proposals that go to verification: the first min(k_verify, block_len - 1)
// (truncated verification; block_len - 1 already holds the R - 1 budget
// cap), cut before the first one whose confidence is below the threshold
// (conf == NULL: no threshold).  Copies the block to the verify layout.
__global__ void draft_limit_kernel(int n, const int32_t* block, int stride_in, const float* conf, int K,
                                   int k_verify, float thr, int32_t* out, int stride_out, int32_t* blen) {
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const int b_in = blen[i];
    int np = min(k_verify, max(b_in - 1, 0));
    if (conf)
      for (int j = 0; j < np; ++j)
        if (conf[(size_t)i * K + j] < thr) { np = j; break; }
    for (int j = 0; j <= k_verify; ++j) out[(size_t)i * stride_out + j] = block[(size_t)i * stride_in + j];
    blen[i] = b_in > 0 ? 1 + np : 0;
  }
  pdl_trigger();
}

// ------------------------------------------------------------------ verification-attention readout
// Alignment Drift §5 / App. D.2: the target's audio attention at one layer,
// averaged over heads, of the block row that produced the next anchor; its
// peak frame centres the drafter's cross-attention window.
// Pass 1, one CTA per (head, request): scores s(f) = q . k_f / sqrt(64) over
// the valid frames (fp32), their max and sum of exp(s - max).
template <typename T>
__global__ void __launch_bounds__(SNT) readout_scores_kernel(int H, const int32_t* req_ids, const int32_t* row,
                                                             const T* q, int d, XKV x, int layer, const int32_t* Fv,
                                                             int max_frames, float* sc, float2* st) {
  __shared__ float sh[SNT + 8];
  __shared__ float qs[WS_DH];
  pdl_wait();
  const int h = blockIdx.x, i = blockIdx.y, heads = gridDim.x;
  const int slot = req_ids[i], F = Fv[slot];
  const int r = min(max(row[i], 0), H - 1);
  if (threadIdx.x < WS_DH) qs[threadIdx.x] = to_f<T>(q[((size_t)i * H + r) * d + h * WS_DH + threadIdx.x]);
  __syncthreads();
  const T* kb = xkv_ptr<T>(x, slot, layer, 0, h, 0);
  float* out = sc + ((size_t)i * heads + h) * max_frames;
  float m = -INFINITY;
  for (int f = threadIdx.x; f < F; f += SNT) {
    const T* kr = kb + (size_t)f * WS_DH;
    float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll 4
    for (int e = 0; e < WS_DH; e += 4) {
      c0 = fmaf(qs[e], to_f<T>(kr[e]), c0);
      c1 = fmaf(qs[e + 1], to_f<T>(kr[e + 1]), c1);
      c2 = fmaf(qs[e + 2], to_f<T>(kr[e + 2]), c2);
      c3 = fmaf(qs[e + 3], to_f<T>(kr[e + 3]), c3);
    }
    const float v = ((c0 + c1) + (c2 + c3)) * 0.125f;
    out[f] = v;
    m = fmaxf(m, v);
  }
  m = block_max<SNT>(m, sh);
  float S = 0.f;
  for (int f = threadIdx.x; f < F; f += SNT) S += expf(out[f] - m);
  S = block_sum<SNT>(S, sh);
  pdl_trigger();
  if (threadIdx.x == 0) st[(size_t)i * heads + h] = make_float2(m, S);
}

// Pass 2, one CTA per request: mean over heads (in head order) of the
// softmax probabilities, argmax over frames (lowest frame on ties).
__global__ void __launch_bounds__(SNT) readout_peak_kernel(int heads, const int32_t* req_ids, const int32_t* Fv,
                                                           int max_frames, const float* sc, const float2* st,
                                                           int32_t* xcenter) {
  __shared__ unsigned long long best[SNT / 32];
  pdl_wait();
  const int i = blockIdx.x, slot = req_ids[i], F = Fv[slot];
  unsigned long long key = 0ull;
  for (int f = threadIdx.x; f < F; f += SNT) {
    float a = 0.f;
    for (int h = 0; h < heads; ++h) {
      const float2 ms = st[(size_t)i * heads + h];
      a += expf(sc[((size_t)i * heads + h) * max_frames + f] - ms.x) / ms.y;
    }
    const unsigned long long k = argmax_key(a / (float)heads, f);
    key = k > key ? k : key;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
    key = other > key ? other : key;
  }
  if ((threadIdx.x & 31) == 0) best[threadIdx.x >> 5] = key;
  __syncthreads();
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int w = 1; w < SNT / 32; ++w) key = best[w] > key ? best[w] : key;
    xcenter[slot] = F > 0 ? argmax_key_id(key) : -1;
  }
}

// Windowed cross-attention of the drafter (Alignment Drift App. A.2: a
// fixed-width mask around a centre frame): rows of request i attend to
// frames max(0, c - w) <= f < min(F, c + w + 1), c = xcenter[slot] (no
// centre yet: every valid frame).  One CTA per (request, head), one warp
// per row; keys in chunks of 64 staged as fp32 in shared memory, online
// softmax in fp32.
template <typename T>
__global__ void __launch_bounds__(128) window_attn_kernel(int H, const int32_t* req_ids, const int32_t* Fv,
                                                          const int32_t* xcenter, int w, const T* Q, int d, XKV x,
                                                          int layer, T* O) {
  __shared__ float Ks[WS_XCHUNK][WS_DH + 1];
  __shared__ float Vs[WS_XCHUNK][WS_DH];
  __shared__ float pw[4][WS_XCHUNK];
  __shared__ float qsh[4][WS_DH];
  pdl_wait();
  const int i = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = req_ids[i], F = Fv[slot], c = xcenter[slot];
  const int lo = c >= 0 ? max(0, c - w) : 0, hi = c >= 0 ? min(F, c + w + 1) : F;
  const T* kb = xkv_ptr<T>(x, slot, layer, 0, h, 0);
  const T* vb = xkv_ptr<T>(x, slot, layer, 1, h, 0);
  // per row: q (2 dims per lane), running max, sum and weighted values
  float qv[4][2], m[4], l[4], a0[4], a1[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = warp + 4 * j;
    m[j] = -INFINITY; l[j] = 0.f; a0[j] = 0.f; a1[j] = 0.f;
    qv[j][0] = qv[j][1] = 0.f;
    if (r < H) {
      qv[j][0] = to_f<T>(Q[((size_t)i * H + r) * d + h * WS_DH + 2 * lane]);
      qv[j][1] = to_f<T>(Q[((size_t)i * H + r) * d + h * WS_DH + 2 * lane + 1]);
    }
  }
  for (int k0 = lo; k0 < hi; k0 += WS_XCHUNK) {
    const int nk = min(WS_XCHUNK, hi - k0);
    __syncthreads();
    for (int e = threadIdx.x; e < nk * WS_DH; e += 128) {
      const int kk = e / WS_DH, dd = e - kk * WS_DH;
      Ks[kk][dd] = to_f<T>(kb[(size_t)(k0 + kk) * WS_DH + dd]);
      Vs[kk][dd] = to_f<T>(vb[(size_t)(k0 + kk) * WS_DH + dd]);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = warp + 4 * j;
      if (r >= H) continue;
      // scores: lane handles keys lane and lane + 32 (the row's query in shared memory)
      qsh[warp][2 * lane] = qv[j][0];
      qsh[warp][2 * lane + 1] = qv[j][1];
      __syncwarp();
      float s[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int kk = lane + 32 * t;
        float acc = 0.f;
        if (kk < nk)
          for (int dd = 0; dd < WS_DH; ++dd) acc = fmaf(qsh[warp][dd], Ks[kk][dd], acc);
        s[t] = kk < nk ? acc * 0.125f : -INFINITY;
      }
      const float mn = fmaxf(m[j], warp_max(fmaxf(s[0], s[1])));
      const float p0 = s[0] > -INFINITY ? expf(s[0] - mn) : 0.f, p1 = s[1] > -INFINITY ? expf(s[1] - mn) : 0.f;
      const float corr = m[j] > -INFINITY ? expf(m[j] - mn) : 0.f;
      l[j] = l[j] * corr + warp_sum(p0 + p1);
      pw[warp][lane] = p0;
      pw[warp][lane + 32] = p1;
      __syncwarp();
      float b0 = 0.f, b1 = 0.f;
      for (int kk = 0; kk < nk; ++kk) {
        b0 = fmaf(pw[warp][kk], Vs[kk][2 * lane], b0);
        b1 = fmaf(pw[warp][kk], Vs[kk][2 * lane + 1], b1);
      }
      __syncwarp();
      a0[j] = a0[j] * corr + b0;
      a1[j] = a1[j] * corr + b1;
      m[j] = mn;
    }
  }
  pdl_trigger();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = warp + 4 * j;
    if (r >= H) continue;
    const float inv = l[j] > 0.f ? 1.f / l[j] : 0.f;
    O[((size_t)i * H + r) * d + h * WS_DH + 2 * lane] = from_f<T>(a0[j] * inv);
    O[((size_t)i * H + r) * d + h * WS_DH + 2 * lane + 1] = from_f<T>(a1[j] * inv);
  }
}

// ------------------------------------------------------------------ acceptance
// One CTA per request.  Whisper-Flash §3.1 / Appendix A.1 / A.4.
__global__ void __launch_bounds__(SNT) accept_kernel(AcceptParams P) {
  __shared__ double cdf_scratch[(SNT / 32) * CDF_SROWS];
  __shared__ float sh[SNT + 8];
  __shared__ int s_emit[17];
  __shared__ int s_ne, s_a, s_stop;
  pdl_wait();
  const ws_accept_args& A = P.a;
  const int i = blockIdx.x;
  const int slot = P.req_ids[i];
  const int blen = A.block_len[i];
  const bool was_done = A.done[i] != 0;
  int R = A.budget[i];
  if (P.tree_n > 0 && threadIdx.x == 0) {       // nothing to commit unless the walk below says so
    P.tpath[(size_t)i * WS_TREE_REC] = P.L[slot];
    P.tpath[(size_t)i * WS_TREE_REC + 1] = 0;
  }
  if (was_done || blen <= 0 || R <= 0) {
    if (threadIdx.x == 0) {
      A.n_acc[i] = 0;
      A.n_emit[i] = 0;
      A.next_len[i] = 0;
      A.next_block[(size_t)i * A.next_stride] = A.block[(size_t)i * A.H];
      if (!was_done && (blen <= 0 || R <= 0)) {
        // an idle request with no budget left is finished
        if (R <= 0) { A.done[i] = 1; if (A.n_done) atomicAdd(A.n_done, 1); }
      }
    }
    return;
  }
  const int32_t* blk = A.block + (size_t)i * A.H;
  // at most R-1 candidates (Appendix A.1); a forced block is taken whole
  int n_prop = A.mode == WS_ACCEPT_FORCED ? blen - 1 : min(blen - 1, max(R - 1, 0));
  n_prop = min(n_prop, A.H - 1);                       // the block holds H tokens
  if (A.mode == WS_ACCEPT_SAMPLE) n_prop = min(n_prop, P.K);   // q rows exist for K candidates
  if (threadIdx.x == 0) { s_ne = 0; s_a = 0; s_stop = 0; }
  __syncthreads();

  // A forced block with a temperature and logits samples its emitted token
  // (the first transcript token of a sampled decode) instead of taking the argmax.
  const bool forced_sample = A.mode == WS_ACCEPT_FORCED && A.temperature > 0.0f && A.p_logits != nullptr;
  if (A.mode == WS_ACCEPT_GREEDY || (A.mode == WS_ACCEPT_FORCED && !forced_sample)) {
    if (threadIdx.x == 0) {
      const int32_t* g = A.target + (size_t)i * A.H;
      int a = 0, ne = 0, last_row = -1;   // last_row: the row whose argmax follows the accepted tokens
      bool eos_hit = false;
      if (A.mode == WS_ACCEPT_FORCED) {
        a = n_prop;
      } else if (P.tree_n > 0) {
        // candidate tree (Alignment Drift App. E.3): from the root, step to the
        // lowest-numbered child whose token is the target's argmax at the
        // current row, at most R - 1 times
        int* rec = P.tpath + (size_t)i * WS_TREE_REC;
        const int rows = min(min(blen, A.H), P.max_pos - P.L[slot]);   // rows whose cache slots exist
        int cur = 0;
        rec[2] = 0;
        while (a < R - 1) {
          int nxt = -1;
          for (int c = cur + 1; c < rows; ++c)
            if ((int)((P.parent4 >> (4 * c)) & 15ull) == cur && blk[c] == g[cur]) { nxt = c; break; }
          if (nxt < 0) break;
          cur = nxt;
          ++a;
          rec[2 + a] = cur;
          s_emit[ne++] = blk[cur];
          if (blk[cur] == P.eos) { eos_hit = true; break; }
        }
        rec[0] = P.L[slot];
        rec[1] = a;
        last_row = cur;
      } else {
        for (int j = 1; j <= n_prop; ++j) {
          if (blk[j] != g[j - 1]) break;
          ++a;
          s_emit[ne++] = blk[j];
          if (blk[j] == P.eos) { eos_hit = true; break; }
        }
      }
      if (!eos_hit) s_emit[ne++] = g[last_row < 0 ? a : last_row];
      s_a = a;
      s_ne = ne;
    }
    __syncthreads();
  } else {
    // Rejection rule: accept y_j iff u_j * q_j(y_j) < p_j(y_j) (FP32).
    const float T = A.temperature;
    if (forced_sample && threadIdx.x == 0) s_a = n_prop;
    for (int j = 1; j <= (forced_sample ? 0 : n_prop); ++j) {
      const int y = blk[j];
      const float* zp = A.p_logits + ((long long)i * A.H + (j - 1)) * P.V;
      const float* zq = A.q_logits + ((long long)i * P.K + (j - 1)) * P.V;
      const float2 ps = P.pstat[(size_t)i * A.H + (j - 1)], qs = P.qstat[(size_t)i * P.K + (j - 1)];
      RowStat sp, sq;
      sp.m = ps.x; sp.S = ps.y;
      sq.m = qs.x; sq.S = qs.y;
      const bool yok = y >= 0 && y < P.V;
      const float py = yok ? expf(scaled(zp, y, T, P.suppress) - sp.m) / sp.S : 0.0f;
      const float qy = yok ? expf(scaled(zq, y, T, P.suppress) - sq.m) / sq.S : 0.0f;
      const float u = ws_uniform(A.seed, (uint32_t)slot, A.round, (uint32_t)j, 1u);
      if (u * qy < py) {
        if (threadIdx.x == 0) { s_emit[s_ne++] = y; s_a = j; if (y == P.eos) s_stop = 1; }
        __syncthreads();
        if (s_stop) break;
        continue;
      }
      // residual (p - q)_+, normalised implicitly by the inverse CDF; p when empty
      auto resid = [&](int v) {
        float pv = expf(scaled(zp, v, T, P.suppress) - sp.m) / sp.S;
        float qv = expf(scaled(zq, v, T, P.suppress) - sq.m) / sq.S;
        return fmaxf(pv - qv, 0.0f);
      };
      // its mass (only whether it is positive matters): eight ids of both
      // rows loaded at once per thread, since the rows stream from HBM
      float r4[4] = {0.f, 0.f, 0.f, 0.f};
      int v = threadIdx.x;
      for (; v + 7 * SNT < P.V; v += 8 * SNT) {
        float zpv[8], zqv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          zpv[q] = __ldg(zp + v + q * SNT);
          zqv[q] = __ldg(zq + v + q * SNT);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int vq = v + q * SNT;
          const float pv = expf(scaled_val(zpv[q], vq, T, P.suppress) - sp.m) / sp.S;
          const float qv = expf(scaled_val(zqv[q], vq, T, P.suppress) - sq.m) / sq.S;
          r4[q & 3] += fmaxf(pv - qv, 0.0f);
        }
      }
      for (; v < P.V; v += SNT) r4[0] += resid(v);
      const float rs = block_sum<SNT>((r4[0] + r4[1]) + (r4[2] + r4[3]), sh);
      const float u2 = ws_uniform(A.seed, (uint32_t)slot, A.round, (uint32_t)j, 2u);
      int tok;
      if (rs > 0.0f) tok = block_inverse_cdf(resid, P.V, u2, cdf_scratch);
      else tok = block_inverse_cdf([&](int v) { return expf(scaled(zp, v, T, P.suppress) - sp.m) / sp.S; }, P.V, u2,
                                   cdf_scratch);
      if (threadIdx.x == 0) { s_emit[s_ne++] = tok; s_stop = 2; }
      __syncthreads();
      break;
    }
    __syncthreads();
    if (s_stop == 0) {   // every candidate accepted: bonus from the target row n_prop
      const float* zp = A.p_logits + ((long long)i * A.H + n_prop) * P.V;
      const float2 ps = P.pstat[(size_t)i * A.H + n_prop];
      RowStat sp;
      sp.m = ps.x; sp.S = ps.y;
      const float u2 = ws_uniform(A.seed, (uint32_t)slot, A.round, (uint32_t)(n_prop + 1), 2u);
      int tok = block_inverse_cdf([&](int v) { return expf(scaled(zp, v, T, P.suppress) - sp.m) / sp.S; }, P.V, u2,
                                  cdf_scratch);
      if (threadIdx.x == 0) s_emit[s_ne++] = tok;
    }
    __syncthreads();
  }

  if (threadIdx.x == 0) {
    const int a = s_a, ne = s_ne;
    P.L[slot] += 1 + a;                 // rollback by length: keep the anchor + a candidates
    R -= ne;
    const int last = s_emit[ne - 1];
    const bool done = (last == P.eos) || R <= 0;
    A.budget[i] = R;
    A.n_acc[i] = a;
    A.n_emit[i] = ne;
    A.next_block[(size_t)i * A.next_stride] = last;
    A.next_len[i] = done ? 0 : 1 + min(P.K, R - 1);
    if (A.transcript) {
      int ol = A.out_len[i];
      for (int k = 0; k < ne; ++k)
        if (ol < A.tcap) A.transcript[(size_t)i * A.tcap + ol++] = s_emit[k];
      A.out_len[i] = ol;
    }
    if (done) {
      A.done[i] = 1;
      if (A.n_done) atomicAdd(A.n_done, 1);
    }
  }
  pdl_trigger();
}

// ------------------------------------------------------------------ candidate trees
// After a tree acceptance, block row j (1 <= j <= a) takes the contents of
// tree row path[j] >= j.  grid (2 * n_layers + 2, n): job x < 2 * n_layers
// moves layer x / 2's keys (x even) or values of cache slots L + path[j] to
// L + j; job 2 * n_layers the history rows; the last job the readout
// queries.  Each thread owns a set of 4-byte words and walks j upwards, so
// a row is read before a later j overwrites it (path[j] >= j).
__global__ void __launch_bounds__(256) tree_commit_kernel(TreeCommit t) {
  pdl_wait();
  const int job = blockIdx.x, i = blockIdx.y;
  const int* rec = t.tpath + (size_t)i * WS_TREE_REC;
  const int slot = t.req_ids[i], L0 = rec[0], a = rec[1];
  const int* path = rec + 2;
  pdl_trigger();
  if (a <= 0) return;
  if (job < 2 * t.n_layers) {
    const int l = job >> 1, kv = job & 1;
    const int nw = WS_DH * t.es / 4;                       // words per head row
    const char* base = t.kv + (size_t)l * t.kv_layer_bytes;
    auto row = [&](int pos, int head) {
      const int page = t.ptab[slot * t.ppr + pos / WS_PAGE];
      const size_t off = (((size_t)page * 2 + kv) * t.heads + head) * (WS_PAGE * WS_DH) + (size_t)(pos % WS_PAGE) * WS_DH;
      return reinterpret_cast<uint32_t*>(const_cast<char*>(base) + off * t.es);
    };
    for (int w = threadIdx.x; w < t.heads * nw; w += blockDim.x) {
      const int head = w / nw, o = w - head * nw;
      for (int j = 1; j <= a; ++j)
        if (path[j] != j) row(L0 + j, head)[o] = row(L0 + path[j], head)[o];
    }
  } else if (job == 2 * t.n_layers) {
    if (!t.hist) return;
    float* h = t.hist + (size_t)slot * t.max_block * t.hist_w;
    for (int w = threadIdx.x; w < t.hist_w; w += blockDim.x)
      for (int j = 1; j <= a; ++j)
        if (path[j] != j) h[(size_t)j * t.hist_w + w] = h[(size_t)path[j] * t.hist_w + w];
  } else {
    if (!t.qread) return;
    const int nw = t.d * t.es / 4;
    uint32_t* q = reinterpret_cast<uint32_t*>(t.qread) + (size_t)i * t.H * nw;
    for (int w = threadIdx.x; w < nw; w += blockDim.x)
      for (int j = 1; j <= a; ++j)
        if (path[j] != j) q[(size_t)j * nw + w] = q[(size_t)path[j] * nw + w];
  }
}

// One CTA per (tree row j, request): row 0 copies the anchor and sets the
// block length (every row of the tree that fits before max_pos; 0 for an
// idle request); row j >= 1 ranks the logits of mask row depth(j) - 1 by
// (value, lower id first) and takes the one of rank rank(j).
__global__ void __launch_bounds__(SNT) tree_tokens_kernel(int n_nodes, unsigned long long depth4,
                                                          unsigned long long rank4, const int32_t* req_ids,
                                                          const int32_t* L, int max_pos, const int32_t* block,
                                                          int stride_in, const float* q, int K, int V, int32_t* out,
                                                          int stride_out, int32_t* blen) {
  __shared__ unsigned long long sk[SNT / 32];
  pdl_wait();
  const int j = blockIdx.x, i = blockIdx.y;
  if (j == 0) {
    pdl_trigger();
    if (threadIdx.x == 0) {
      out[(size_t)i * stride_out] = block[(size_t)i * stride_in];
      const int b_in = blen[i];
      blen[i] = b_in > 0 ? max(1, min(n_nodes, max_pos - L[req_ids[i]])) : 0;
    }
    return;
  }
  const int depth = tree_depth(depth4, j), rank = (int)((rank4 >> (4 * j)) & 15ull);
  const float* z = q + ((long long)i * K + (depth - 1)) * V;
  unsigned long long prev = ~0ull;
  for (int r = 0; r <= rank; ++r) {
    unsigned long long best = 0ull;
    for (int v = threadIdx.x; v < V; v += SNT) {
      const unsigned long long k = argmax_key(z[v], v);
      if (k < prev && k > best) best = k;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sk[threadIdx.x >> 5] = best;
    __syncthreads();
    best = 0ull;
#pragma unroll
    for (int w = 0; w < SNT / 32; ++w) best = sk[w] > best ? sk[w] : best;
    prev = best;
  }
  pdl_trigger();
  if (threadIdx.x == 0) out[(size_t)i * stride_out + j] = argmax_key_id(prev);
}

// ------------------------------------------------------------------ synthetic drafts
__global__ void draft_synth_kernel(int K, const int32_t* req_ids, const int32_t* L, int32_t* block,
                                   const int32_t* traj, int tlen, const uint8_t* cmask, const int32_t* ctok,
                                   int max_pos) {
  pdl_wait();
  const int i = blockIdx.x, j = threadIdx.x + 1;
  if (j > K) return;
  const int t = min(L[req_ids[i]], max_pos - 1);
  const size_t c = ((size_t)i * max_pos + t) * K + (j - 1);
  int tok;
  if (cmask[c] || t + j >= tlen) tok = ctok[c];
  else tok = traj[(size_t)i * tlen + t + j];
  block[(size_t)i * (K + 1) + j] = tok;
  pdl_trigger();
}

}  // namespace

// ------------------------------------------------------------------ launchers
template <typename T>
cudaError_t launch_embed_target(int n, int H, const RowMap& rm, unsigned long long depth4, const int32_t* block,
                                const T* E, const T* P, int d, int V, float* x, int32_t* pend_start, int32_t* pend_n,
                                int32_t* status, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n * H), dim3(128), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, embed_target_kernel<T>, rm, depth4, block, E, P, d, V, x, pend_start, pend_n,
                            status);
}
template <typename T>
cudaError_t launch_embed_draft(int n, int K1, const int32_t* req_ids, const int32_t* block, const T* E, const T* m,
                               int d, int V, float* x, int32_t* pend_n, int32_t* status, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n * K1), dim3(128), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, embed_draft_kernel<T>, K1, req_ids, block, E, m, d, V, x, pend_n, status);
}
template <typename T>
cudaError_t launch_layernorm(int M, int d, const float* x, int ldx, const T* g, const T* b, T* y, int ldy,
                             int group_skip, cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (d % 128 != 0 || d > 2048) return cudaErrorInvalidValue;
  cudaLaunchAttribute at[1];
  if (M >= LN_MANY) {
    cudaLaunchConfig_t cfg = make_cfg(dim3((M + 4 * LN_RPW - 1) / (4 * LN_RPW)), dim3(128), 0, s, pdl, at);
    ws_count_launches(1);
    return cudaLaunchKernelEx(&cfg, d <= 1280 ? layernorm_rows_kernel<T, 10> : layernorm_rows_kernel<T, 16>, M, d, x,
                              ldx, g, b, y, ldy, group_skip);
  }
  cudaLaunchConfig_t cfg = make_cfg(dim3((M + 3) / 4), dim3(128), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, d <= 1280 ? layernorm_kernel<T, 10> : layernorm_kernel<T, 16>, M, d, x, ldx, g, b, y,
                            ldy, group_skip);
}
cudaError_t launch_argmax_init(int M, unsigned long long* keys, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((M + 255) / 256), dim3(256), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, argmax_init_kernel, M, keys);
}
cudaError_t launch_argmax_finalize(int n, int H, const int32_t* block_len, const unsigned long long* keys,
                                   int32_t* out, int out_stride, int out_col0, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((n * H + 255) / 256), dim3(256), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, argmax_finalize_kernel, n, H, block_len, keys, out, out_stride, out_col0);
}
template <typename T>
cudaError_t launch_hist_gather(int n, int Hp, const int32_t* req_ids, const int32_t* pend_n, const float* hist,
                               int max_block, int n_hist, int d, T* feat, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n * Hp), dim3(256), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, hist_gather_kernel<T>, Hp, req_ids, pend_n, hist, max_block, n_hist, d, feat);
}
cudaError_t launch_rope_table(float* tab, int max_pos, cudaStream_t s) {
  int n = max_pos * (WS_DH / 2);
  ws_count_launches(1);
  rope_table_kernel<<<(n + 255) / 256, 256, 0, s>>>(tab, max_pos);
  return cudaGetLastError();
}
cudaError_t launch_set_frames(int n, const int32_t* req_ids, const int32_t* cu, const int32_t* valid,
                              int max_frames, int32_t* Fc, int32_t* Fv, int32_t* status, cudaStream_t s) {
  ws_count_launches(1);
  set_frames_kernel<<<(n + 127) / 128, 128, 0, s>>>(n, req_ids, cu, valid, max_frames, Fc, Fv, status);
  return cudaGetLastError();
}
cudaError_t launch_reset(int n, const int32_t* req_ids, int32_t* L, int32_t* pend_n, int32_t* xcenter,
                         cudaStream_t s) {
  ws_count_launches(1);
  reset_kernel<<<(n + 127) / 128, 128, 0, s>>>(n, req_ids, L, pend_n, xcenter);
  return cudaGetLastError();
}
template <typename T>
cudaError_t launch_readout(int n, int H, const int32_t* req_ids, const int32_t* row, const T* q, int d, const XKV& x,
                           int layer, const int32_t* Fv, int max_frames, float* sc, float2* st, int32_t* xcenter,
                           cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  const int heads = d / WS_DH;
  cudaLaunchConfig_t cfg = make_cfg(dim3(heads, n), dim3(SNT), 0, s, pdl, at);
  ws_count_launches(2);
  cudaError_t e = cudaLaunchKernelEx(&cfg, readout_scores_kernel<T>, H, req_ids, row, q, d, x, layer, Fv, max_frames,
                                     sc, st);
  if (e != cudaSuccess) return e;
  cfg = make_cfg(dim3(n), dim3(SNT), 0, s, pdl, at);
  return cudaLaunchKernelEx(&cfg, readout_peak_kernel, heads, req_ids, Fv, max_frames, (const float*)sc,
                            (const float2*)st, xcenter);
}
template cudaError_t launch_readout<float>(int, int, const int32_t*, const int32_t*, const float*, int, const XKV&,
                                           int, const int32_t*, int, float*, float2*, int32_t*, cudaStream_t, bool);
template cudaError_t launch_readout<bf16>(int, int, const int32_t*, const int32_t*, const bf16*, int, const XKV&, int,
                                          const int32_t*, int, float*, float2*, int32_t*, cudaStream_t, bool);

template <typename T>
cudaError_t launch_window_attn(int n, int H, const int32_t* req_ids, const int32_t* Fv, const int32_t* xcenter, int w,
                               const T* Q, int d, const XKV& x, int layer, T* O, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n, d / WS_DH), dim3(128), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, window_attn_kernel<T>, H, req_ids, Fv, xcenter, w, Q, d, x, layer, O);
}
template cudaError_t launch_window_attn<float>(int, int, const int32_t*, const int32_t*, const int32_t*, int,
                                               const float*, int, const XKV&, int, float*, cudaStream_t, bool);
template cudaError_t launch_window_attn<bf16>(int, int, const int32_t*, const int32_t*, const int32_t*, int,
                                              const bf16*, int, const XKV&, int, bf16*, cudaStream_t, bool);

cudaError_t launch_draft_limit(int n, int K, const int32_t* block, int stride_in, const float* q, int V, float T,
                               const uint32_t* sup, float* conf, int k_verify, float thr, int32_t* out,
                               int stride_out, int32_t* blen, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaError_t e = cudaSuccess;
  if (thr > 0.0f && min(K, k_verify) > 0) {
    cudaLaunchConfig_t cfg = make_cfg(dim3(min(K, k_verify), n), dim3(SNT), 0, s, pdl, at);
    ws_count_launches(1);
    e = cudaLaunchKernelEx(&cfg, draft_conf_kernel, block, stride_in, q, K, V, T, sup, conf);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = make_cfg(dim3((n + 127) / 128), dim3(128), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, draft_limit_kernel, n, block, stride_in, thr > 0.0f ? (const float*)conf : nullptr,
                            K, k_verify, thr, out, stride_out, blen);
}

cudaError_t launch_get_lengths(int n, const int32_t* req_ids, const int32_t* L, int32_t* out, cudaStream_t s) {
  ws_count_launches(1);
  get_lengths_kernel<<<(n + 127) / 128, 128, 0, s>>>(n, req_ids, L, out);
  return cudaGetLastError();
}
cudaError_t launch_sample_rows(int n, int rows, const int32_t* req_ids, const float* logits, long long row_stride,
                               int V, float T, uint64_t seed, uint64_t rnd, const uint32_t* suppress, int32_t* out,
                               int out_stride, int out_col0, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n * rows), dim3(SNT), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, sample_rows_kernel, rows, req_ids, logits, row_stride, V, T, seed, rnd,
                            suppress, out, out_stride, out_col0);
}
cudaError_t launch_accept(int n, const AcceptParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  const ws_accept_args& a = p.a;
  const bool sampling = a.p_logits && a.temperature > 0.0f &&
                        (a.mode == WS_ACCEPT_SAMPLE || a.mode == WS_ACCEPT_FORCED);
  if (sampling) {
    cudaLaunchConfig_t c1 = make_cfg(dim3(n * a.H), dim3(SNT), 0, s, pdl, at);
    ws_count_launches(1);
    cudaError_t e = cudaLaunchKernelEx(&c1, row_stats_kernel, (const float*)a.p_logits, a.H, p.V, a.temperature,
                                       p.suppress, p.pstat);
    if (e != cudaSuccess) return e;
    if (a.mode == WS_ACCEPT_SAMPLE) {
      cudaLaunchConfig_t c2 = make_cfg(dim3(n * p.K), dim3(SNT), 0, s, pdl, at);
      ws_count_launches(1);
      e = cudaLaunchKernelEx(&c2, row_stats_kernel, (const float*)a.q_logits, p.K, p.V, a.temperature, p.suppress,
                             p.qstat);
      if (e != cudaSuccess) return e;
    }
  }
  cudaLaunchConfig_t cfg = make_cfg(dim3(n), dim3(SNT), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, accept_kernel, p);
}
cudaError_t launch_tree_commit(int n, const TreeCommit& t, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(2 * t.n_layers + 2, n), dim3(256), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, tree_commit_kernel, t);
}
cudaError_t launch_tree_tokens(int n, int n_nodes, unsigned long long depth4, unsigned long long rank4,
                               const int32_t* req_ids, const int32_t* L, int max_pos, const int32_t* block,
                               int stride_in, const float* q, int K, int V, int32_t* out, int stride_out,
                               int32_t* blen, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n_nodes, n), dim3(SNT), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, tree_tokens_kernel, n_nodes, depth4, rank4, req_ids, L, max_pos, block, stride_in,
                            q, K, V, out, stride_out, blen);
}
cudaError_t launch_draft_synth(int n, int K, const int32_t* req_ids, const int32_t* L, int32_t* block,
                               const int32_t* traj, int tlen, const uint8_t* cmask, const int32_t* ctok, int max_pos,
                               cudaStream_t s, bool pdl) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n), dim3(32), 0, s, pdl, at);
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, draft_synth_kernel, K, req_ids, L, block, traj, tlen, cmask, ctok, max_pos);
}

#define INST(T)                                                                                                     \
  template cudaError_t launch_embed_target<T>(int, int, const RowMap&, unsigned long long, const int32_t*, const T*,  \
                                              const T*, int, int,                                                    \
                                              float*, int32_t*, int32_t*, int32_t*, cudaStream_t, bool);             \
  template cudaError_t launch_embed_draft<T>(int, int, const int32_t*, const int32_t*, const T*, const T*, int, int, \
                                             float*, int32_t*, int32_t*, cudaStream_t, bool);                        \
  template cudaError_t launch_layernorm<T>(int, int, const float*, int, const T*, const T*, T*, int, int,           \
                                           cudaStream_t, bool);                                                      \
  template cudaError_t launch_hist_gather<T>(int, int, const int32_t*, const int32_t*, const float*, int, int, int, \
                                             T*, cudaStream_t, bool);
INST(float)
INST(bf16)
