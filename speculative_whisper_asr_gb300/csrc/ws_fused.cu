// Persistent block verification for small blocks (at most 16 query rows in
// one call): the whole target pass of ws_verify -- token + position
// embedding, every decoder layer (Whisper-Flash §3.1: the target scores all
// K+1 block rows in one forward), final layer norm, tied LM head and argmax
// -- in one cooperative kernel with one CTA per SM.
//
// Why one kernel: at batch 1 a verify step streams ~1.9 GB of weights and
// acoustic keys/values but is a chain of ~400 small dependent operations.
// As separate kernels each one pays its launch, its ramp-up (first HBM
// bytes) and its drain.  Here the work is laid out per CTA in a static
// schedule:
//   * warp 0 streams every weight tile (128 rows x 64 k, TMA, 128-byte
//     swizzle) and every acoustic key/value chunk this CTA will consume, in
//     consumption order, through a ring of shared-memory slots.  It waits
//     only for a free slot, so HBM reads run ahead across stage and layer
//     boundaries;
//   * warps 1..7 run the stages one after another, separated by grid-wide
//     barriers: GEMM stages (layer-norm or activation rows written straight
//     into the swizzled B operand, tcgen05.mma into TMEM, split-K partials
//     folded in split order by the tile's last-arriving CTA, fused
//     epilogue) and attention stages (one (request, head, 64-key split) unit
//     at a time, partial softmax, folded by the group's last arriver).
//
// The arithmetic is that of the per-op path: the same split-K factors and
// k order, the same warp layer norm, attention update and fold, and the same
// epilogues, so both give bit-identical rows.  Every wait is bounded: a
// timeout sets the device status word and the kernel winds down (waiting,
// again bounded, for its own copies in flight) instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "ws_attn_common.cuh"
#include "ws_attn_mma.cuh"
#include "ws_epilogue.cuh"
#include "ws_fused.cuh"
#include "ws_tc.cuh"

namespace {

using namespace tc;

constexpr int NT = 256;              // threads: warp 0 streams, warps 1..7 compute
constexpr int NCW = 7;               // compute warps
constexpr int NCT = NCW * 32;        // compute threads
constexpr int FIRST_EPI_WARP = 4;    // warps 4..7 read TMEM lane quarters 0..3
constexpr int MAXR = FUSED_MAX_ROWS;
constexpr int SLOT = A_BYTES;        // ring slot: one 128 x 64 bf16 weight tile (16 KB)
constexpr int KV_HALF = SLOT / 2;    // acoustic chunk: K at +0, V at +8 KB (64 keys x 64 dims bf16 each)
constexpr int BKB = MAXR * 128;      // B operand bytes per k-block: 16 rows x 128 B
constexpr uint32_t IDESC = idesc_bf16(BM, MAXR);
constexpr uint32_t TMEM_COLS = 32;
constexpr long long SPIN_BUDGET = 1ll << 31;   // clock cycles (~1 s) before a grid barrier gives up
constexpr int LN_MAXV = 10;          // layer-norm rows up to d = 1280 in 10 float4 per lane

// attention scratch inside the work region: one chunk of keys and values (bf16)
constexpr int ATT_K = 0;
constexpr int ATT_V = ATT_K + WS_XCHUNK * WS_DH * 2;
constexpr int ATT_BYTES = ATT_V + WS_XCHUNK * WS_DH * 2;

__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void compute_sync() { named_sync(1, NCT); }
__device__ __forceinline__ void epi_sync() { named_sync(2, 128); }

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct Shared {
  uint64_t full[FUSED_MAX_RING], empty[FUSED_MAX_RING], mma_done, la_bar;
  uint32_t tmem_base;
  int flag;                          // last-arriver broadcast
  int ok;                            // grid barrier outcome
  int abort;                         // a wait of this CTA ran out
  uint32_t issued;                   // ring items the producer issued
  unsigned long long keys[4][MAXR];  // LM head: per-epilogue-warp row maxima
  // rows of this call: request slot, block row, position, K/V-writable, cache page
  int row_slot[MAXR], row_j[MAXR], row_pos[MAXR], row_valid[MAXR], row_page[MAXR];
};

// Grid-wide barrier of the compute warps (sense reversal on a generation
// word; the arrival count resets itself).  False when the wait ran out.
__device__ bool grid_sync(const FusedArgs& a, Shared& sh) {
  compute_sync();
  if (threadIdx.x == 32) {
    bool ok = true;
    unsigned* count = a.gbar;
    unsigned* gen = a.gbar + 1;
    const unsigned g = ld_acquire(gen);
    __threadfence();
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
      atomicExch(count, 0u);
      __threadfence();
      st_release(gen, g + 1u);
    } else {
      const long long t0 = clock64();
      while (ld_acquire(gen) == g) {
        if (clock64() - t0 > SPIN_BUDGET) { ok = false; atomicOr(a.status, WS_ST_TIMEOUT); break; }
      }
    }
    __threadfence();
    sh.ok = ok;
  }
  compute_sync();
  return sh.ok != 0;
}

__device__ __forceinline__ void split_range(int kb_total, int splits, int sp, int& kb0, int& kb1) {
  kb0 = (int)((long long)sp * kb_total / splits);
  kb1 = (int)((long long)(sp + 1) * kb_total / splits);
}

__device__ __forceinline__ int stage_units(const FusedArgs& a, const FusedStage& st) {
  if (st.kind == FS_GEMM) return ((st.N + BM - 1) / BM) * st.splits;
  if (st.kind == FS_SELF) return a.n * a.heads * a.nsplit_self;
  if (st.kind == FS_CROSS) return a.n * a.heads * a.nsplit_cross;
  return 0;
}

// Units of consecutive stages are dealt round-robin across the CTAs: stage
// g's unit u runs on CTA (u + off_g) mod G, off_g = units of the stages
// before it.  Every CTA then gets about the same share of every layer's
// weight tiles, and its ring can be filled ahead through stages in which it
// has little or no work.
__device__ __forceinline__ int first_unit(int off) {
  const int G = gridDim.x;
  return (int)((blockIdx.x + G - off % G) % G);
}

// ------------------------------------------------------------------ producer (warp 0, lane 0)
__device__ void producer(const FusedArgs& a, uint8_t* ring, Shared& sh) {
  const int G = gridDim.x, R = a.ring_slots;
  uint32_t it = 0;
  int off = 0;
  for (int g = 0; g < a.n_stages; ++g) {
    const FusedStage& st = a.stages[g];
    const int units = stage_units(a, st);
    const int u0 = first_unit(off);
    off += units;
    if (st.kind != FS_GEMM && st.kind != FS_CROSS) continue;
    for (int u = u0; u < units; u += G) {
      int kb0 = 0, kb1 = 1, tile = 0;
      if (st.kind == FS_GEMM) {
        tile = u / st.splits;
        split_range(st.kb_total, st.splits, u - tile * st.splits, kb0, kb1);
      }
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = (int)(it % (uint32_t)R);
        const uint32_t ph = (it / (uint32_t)R) & 1u;
        if (!mbar_wait(&sh.empty[s], ph ^ 1u)) {
          atomicOr(a.status, WS_ST_TIMEOUT);
          sh.issued = it;
          return;
        }
        uint8_t* dst = ring + (size_t)s * SLOT;
        if (st.kind == FS_GEMM) {
          mbar_expect_tx(&sh.full[s], SLOT);
          tma_load_2d(dst, reinterpret_cast<const CUtensorMap*>(st.map), &sh.full[s], kb * BK, tile * BM);
        } else {
          // acoustic keys / values of unit (i, head, split): rows [k_lo, k_lo + nk)
          const int per_req = a.heads * a.nsplit_cross;
          const int i = u / per_req, rem = u - i * per_req, head = rem / a.nsplit_cross;
          const int sp = rem - head * a.nsplit_cross;
          const int slot = a.req_ids[i];
          const int k_lo = sp * WS_XCHUNK;
          const int nk = max(0, min(a.Fv[slot] - k_lo, WS_XCHUNK));
          if (nk > 0) {
            const uint32_t bytes = (uint32_t)(nk * WS_DH * 2);
            mbar_expect_tx(&sh.full[s], 2 * bytes);
            bulk_g2s(dst, xkv_ptr<bf16>(a.xkv, slot, st.layer, 0, head, k_lo), bytes, &sh.full[s]);
            bulk_g2s(dst + KV_HALF, xkv_ptr<bf16>(a.xkv, slot, st.layer, 1, head, k_lo), bytes, &sh.full[s]);
          } else {
            mbar_arrive(&sh.full[s]);
          }
        }
      }
    }
  }
  sh.issued = it;
}

// Before exit: every copy this CTA issued has landed (bounded), also after
// an aborted run in which the computation stopped consuming.
__device__ void drain(const FusedArgs& a, Shared& sh) {
  const uint32_t R = (uint32_t)a.ring_slots, n = sh.issued;
  const uint32_t first = n > R ? n - R : 0u;
  for (uint32_t it = first; it < n; ++it) {
    const int s = (int)(it % R);
    if (!mbar_wait(&sh.full[s], (it / R) & 1u)) { atomicOr(a.status, WS_ST_TIMEOUT); break; }
  }
}

// ------------------------------------------------------------------ GEMM stage
// B operand of one unit: rows 0..15 x k-blocks [kb0, kb0 + nkb) in the layout
// a TMA box of 16 rows x 64 bf16 with 128-byte swizzle has: row r at byte
// r * 128 of its k-block, 16-byte chunk c stored at chunk c ^ (r & 7).
__device__ __forceinline__ uint32_t b_offset(int r, int chunk) {
  return (uint32_t)(r * 128 + ((chunk ^ (r & 7)) << 4));
}

__device__ void build_b(const FusedArgs& a, const FusedStage& st, int kb0, int nkb, uint8_t* bbuf) {
  const int tid = threadIdx.x - 32, warp = tid >> 5;
  const int M = a.M;
  for (int idx = tid; idx < (MAXR - M) * nkb * 8; idx += NCT) {   // rows M..15 are zero
    const int r = M + idx / (nkb * 8), rem = idx % (nkb * 8), j = rem >> 3, c = rem & 7;
    *reinterpret_cast<uint4*>(bbuf + j * BKB + b_offset(r, c)) = make_uint4(0u, 0u, 0u, 0u);
  }
  const int k_lo = kb0 * BK, k_hi = (kb0 + nkb) * BK;
  if (st.in_kind == FIN_LN) {
    for (int r = warp; r < M; r += NCW) {
      const float* xs[1] = {a.x + (size_t)r * a.d};
      auto put = [&](int, int k, float v0, float v1, float v2, float v3) {
        if (k < k_lo || k >= k_hi) return;
        const int kl = k - k_lo, j = kl >> 6, col = kl & 63;
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v0, v1);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(v2, v3);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t*>(&p0);
        w.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(bbuf + j * BKB + b_offset(r, col >> 3) + (col & 7) * 2) = w;
      };
      if (a.d <= 128 * LN_MAXV) ln_rows_warp<true, 1, LN_MAXV>(xs, 1, a.d, st.ln_g, st.ln_b, true, put);
      else ln_rows_warp<true, 1, 16>(xs, 1, a.d, st.ln_g, st.ln_b, true, put);
    }
  } else {
    for (int idx = tid; idx < M * nkb * 8; idx += NCT) {
      const int r = idx / (nkb * 8), rem = idx % (nkb * 8), j = rem >> 3, c = rem & 7;
      const uint4 v =
          __ldcg(reinterpret_cast<const uint4*>(st.act + (size_t)r * st.ld_act + k_lo + j * BK + c * 8));
      *reinterpret_cast<uint4*>(bbuf + j * BKB + b_offset(r, c)) = v;
    }
  }
  fence_async_smem();      // generic-proxy writes -> visible to the tensor core
}

__device__ Epi stage_epi(const FusedArgs& a, const FusedStage& st) {
  Epi e;
  memset(&e, 0, sizeof e);
  e.kind = st.epi;
  e.d = a.d;
  e.status = a.status;
  e.suppress = a.suppress;
  e.max_block = a.max_block;
  e.bias = st.bias;
  e.bias2 = st.bias2;
  e.out = st.out;
  e.ldo = st.ldo;
  e.rm = a.rm;
  if (st.epi == EPI_QKV) {
    e.kv.base = a.kv + (size_t)st.layer * a.kv_layer_bytes;
    e.kv.ptab = a.ptab;
    e.kv.ppr = a.ppr;
    e.kv.n_heads = a.heads;
  } else if (st.epi == EPI_RESID) {
    e.resid = a.x;
    e.ldr = a.d;
    if (st.hist_idx >= 0) { e.hist = a.hist; e.hist_idx = st.hist_idx; e.n_hist = a.n_hist; }
  } else if (st.epi == EPI_LOGITS) {
    e.logits = a.logits;
    e.ldl = a.V;
    e.amax = a.amax;
  }
  return e;
}

// Epilogue of one feature n for rows 0 .. M-1 (v[c] = row c), per element the
// arithmetic of epi_pair; row facts come from the shared row table and all
// residual reads are issued together.
__device__ void fused_epilogue(const FusedArgs& a, const FusedStage& st, int n, const float* v, const Shared& sh) {
  if (n >= st.N) return;
  const int M = a.M, d = a.d;
  switch (st.epi) {
    case EPI_RESID: {
      const float b = bias_at<bf16>(st.bias, n);
      float xr[MAXR];
#pragma unroll
      for (int c = 0; c < MAXR; ++c)
        if (c < M) xr[c] = __ldcg(a.x + (size_t)c * d + n);
#pragma unroll
      for (int c = 0; c < MAXR; ++c) {
        if (c < M) {
          const float val = xr[c] + (v[c] + b);
          a.x[(size_t)c * d + n] = val;
          if (st.hist_idx >= 0)
            a.hist[(((size_t)sh.row_slot[c] * a.max_block + sh.row_j[c]) * a.n_hist + st.hist_idx) * d + n] = val;
        }
      }
      break;
    }
    case EPI_QKV: {
      const int part = n / d, nn = n - part * d;
      if (part == 0) {
        const float b = bias_at<bf16>(st.bias, nn);
#pragma unroll
        for (int c = 0; c < MAXR; ++c)
          if (c < M) a.q[(size_t)c * d + nn] = __float2bfloat16_rn(v[c] + b);
      } else {
        const float b = part == 2 ? bias_at<bf16>(st.bias2, nn) : 0.0f;
        bf16* pool = reinterpret_cast<bf16*>(a.kv + (size_t)st.layer * a.kv_layer_bytes);
        const int head = nn / WS_DH, dd = nn % WS_DH;
#pragma unroll
        for (int c = 0; c < MAXR; ++c) {
          if (c < M && sh.row_valid[c]) {
            const size_t off = (((size_t)sh.row_page[c] * 2 + (part - 1)) * a.heads + head) * (WS_PAGE * WS_DH) +
                               (size_t)(sh.row_pos[c] % WS_PAGE) * WS_DH + dd;
            pool[off] = __float2bfloat16_rn(part == 2 ? v[c] + b : v[c]);
          }
        }
      }
      break;
    }
    case EPI_STORE:
    case EPI_GELU: {
      const float b = bias_at<bf16>(st.bias, n);
      bf16* out = reinterpret_cast<bf16*>(st.out);
#pragma unroll
      for (int c = 0; c < MAXR; ++c) {
        if (c < M) {
          float val = v[c] + b;
          if (st.epi == EPI_GELU) val = gelu_erf(val);
          out[(size_t)c * st.ldo + n] = __float2bfloat16_rn(val);
        }
      }
      break;
    }
    default:        // LOGITS has its own epilogue; no other kind occurs in the verify pass
      break;
  }
}

// LM head epilogue: the logit values of epi_columns16; the argmax keys are
// reduced over the four epilogue warps before one atomicMax per row.
__device__ void logits_epilogue(const FusedArgs& a, const Epi& e, int N, int n, const float* v, Shared& sh) {
  const int lane = threadIdx.x & 31, ew = (threadIdx.x >> 5) - FIRST_EPI_WARP;
#pragma unroll
  for (int c = 0; c < MAXR; ++c) {
    unsigned long long key = 0ull;
    if (c < a.M && n < N) {
      const float y = epi_logit(e, n, v[c]);
      if (e.logits) e.logits[(long long)c * e.ldl + n] = y;
      key = argmax_key(y, n);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
      key = other > key ? other : key;
    }
    if (lane == 0) sh.keys[ew][c] = key;
  }
  epi_sync();
  const int c = threadIdx.x - FIRST_EPI_WARP * 32;
  if (c < a.M) {
    unsigned long long k = sh.keys[0][c];
    for (int w = 1; w < 4; ++w) k = sh.keys[w][c] > k ? sh.keys[w][c] : k;
    if (k != 0ull) atomicMax(a.amax + c, k);
  }
}

__device__ void gemm_stage(const FusedArgs& a, const FusedStage& st, int u0, uint8_t* ring, uint8_t* work,
                           Shared& sh, uint32_t& it, uint32_t& done_ph, uint32_t& la_ph) {
  const int G = gridDim.x, R = a.ring_slots;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = stage_units(a, st);
  const uint32_t tmem = sh.tmem_base;
  const Epi e = stage_epi(a, st);
  int built0 = -1, builtn = -1;
  for (int u = u0; u < units; u += G) {
    const int tile = u / st.splits, sp = u - tile * st.splits;
    int kb0, kb1;
    split_range(st.kb_total, st.splits, sp, kb0, kb1);
    const int nkb = kb1 - kb0;
    if (kb0 != built0 || nkb != builtn) {       // the LM head reuses one B operand for all its tiles
      build_b(a, st, kb0, nkb, work);
      built0 = st.splits == 1 ? kb0 : -1;      // a split-K fold reuses the work region
      builtn = nkb;
    }
    compute_sync();
    if (sh.abort) return;
    if (threadIdx.x == 32) {
      // ---- MMA issuer: weights from the ring, activation rows from the B operand
      for (int j = 0; j < nkb; ++j) {
        const uint32_t ii = it + (uint32_t)j;
        const int s = (int)(ii % (uint32_t)R);
        if (!mbar_wait(&sh.full[s], (ii / (uint32_t)R) & 1u)) {
          atomicOr(a.status, WS_ST_TIMEOUT);
          sh.abort = 1;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sdesc_sw128(smem_u32(ring + (size_t)s * SLOT));
        const uint64_t bd = sdesc_sw128(smem_u32(work + j * BKB));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), IDESC, (j | kk) != 0 ? 1u : 0u);
        umma_commit(&sh.empty[s]);
      }
      umma_commit(&sh.mma_done);
    }
    it += (uint32_t)nkb;
    if (warp >= FIRST_EPI_WARP) {
      const int quarter = warp - FIRST_EPI_WARP;
      const int fl = quarter * 32 + lane;      // feature within the tile (TMEM lane)
      const int n = tile * BM + fl;
      float v[MAXR];
      if (!mbar_wait(&sh.mma_done, done_ph)) { atomicOr(a.status, WS_ST_TIMEOUT); sh.abort = 1; }
      tc_fence_after();
      tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16), v);
      if (st.splits == 1) {
        if (st.epi == EPI_LOGITS) logits_epilogue(a, e, st.N, n, v, sh);
        else fused_epilogue(a, st, n, v, sh);
      } else {
        // split-K: park the partial; the tile's last arriver pulls every split's
        // partial into shared memory with bulk copies (one round trip for all
        // of them) and adds them in split order
        float* p = a.part + (size_t)(tile * st.splits + sp) * MAXR * BM + fl;
        for (int c = 0; c < a.M; ++c) p[c * BM] = v[c];
        fence_async_global();     // read back through the async proxy
        __threadfence();
        epi_sync();
        if (threadIdx.x == FIRST_EPI_WARP * 32) {
          const int old = atomicAdd(a.tile_ctr + tile, 1);
          const int last = old == st.splits - 1;
          if (last) a.tile_ctr[tile] = 0;
          sh.flag = last;
        }
        epi_sync();
        if (sh.flag) {
          const uint32_t bytes = (uint32_t)(a.M * BM * 4);
          const int per_pass = max(1, (int)(a.work_bytes / bytes));
          const float* base = a.part + (size_t)tile * st.splits * MAXR * BM;
          float* buf = reinterpret_cast<float*>(work);
          for (int s0 = 0; s0 < st.splits; s0 += per_pass) {
            const int ns = min(per_pass, st.splits - s0);
            if (threadIdx.x == FIRST_EPI_WARP * 32) {
              __threadfence();
              fence_async_global();
              mbar_expect_tx(&sh.la_bar, (uint32_t)ns * bytes);
              for (int q = 0; q < ns; ++q)
                bulk_g2s(buf + (size_t)q * a.M * BM, base + (size_t)(s0 + q) * MAXR * BM, bytes, &sh.la_bar);
            }
            if (!mbar_wait(&sh.la_bar, la_ph)) { atomicOr(a.status, WS_ST_TIMEOUT); sh.abort = 1; }
            la_ph ^= 1u;
            for (int q = 0; q < ns; ++q) {
              const float* ps = buf + (size_t)q * a.M * BM + fl;
#pragma unroll
              for (int c = 0; c < MAXR; ++c) {
                if (c < a.M) {
                  if (s0 + q == 0) v[c] = ps[c * BM];
                  else v[c] += ps[c * BM];
                }
              }
            }
            epi_sync();          // the buffer is refilled by the next pass
          }
          if (st.epi == EPI_LOGITS) logits_epilogue(a, e, st.N, n, v, sh);   // an LM head of < 100 tiles splits K
          else fused_epilogue(a, st, n, v, sh);
        }
      }
      tc_fence_before();
    }
    done_ph ^= 1u;
    compute_sync();      // TMEM and the B operand are free for the next unit
  }
}

// ------------------------------------------------------------------ attention stages
// Self: keys 0 .. L + j of the paged cache for row j (the block's own keys
// were written by this layer's QKV stage).  Cross: the request's valid
// acoustic frames, chunk staged by the producer.
__device__ void attn_stage(const FusedArgs& a, const FusedStage& st, int u0, uint8_t* ring, uint8_t* work,
                           Shared& sh, uint32_t& it) {
  const bool cross = st.kind == FS_CROSS;
  const int G = gridDim.x, R = a.ring_slots;
  const int tid = threadIdx.x - 32, warp = tid >> 5, lane = threadIdx.x & 31;
  const int nsplit = cross ? a.nsplit_cross : a.nsplit_self;
  const int per_req = a.heads * nsplit;
  const int units = a.n * per_req;
  const int H = a.H;
  for (int u = u0; u < units; u += G) {
    const int i = u / per_req, rem = u - i * per_req, head = rem / nsplit, sp = rem - head * nsplit;
    const int slot = a.req_ids[i];
    const int k_lo = sp * WS_XCHUNK;
    int k_hi, nrow = H, Lr = 0;
    if (!cross) {
      Lr = a.rm.L[slot];
      nrow = min(a.block_len[i], H);
      k_hi = min(min(Lr + nrow, a.max_pos), k_lo + WS_XCHUNK);
    } else {
      k_hi = min(a.Fv[slot], k_lo + WS_XCHUNK);
    }
    const int nk = max(0, k_hi - k_lo);
    // keys / values of the chunk as linear [key][64] bf16 rows: the producer's
    // ring slot (acoustic) or copied from the paged cache (self)
    uint8_t* Ks = work + ATT_K;
    uint8_t* Vs = work + ATT_V;
    int s = -1;
    if (cross) {
      s = (int)(it % (uint32_t)R);
      if (!mbar_wait(&sh.full[s], (it / (uint32_t)R) & 1u)) { atomicOr(a.status, WS_ST_TIMEOUT); sh.abort = 1; }
      Ks = ring + (size_t)s * SLOT;
      Vs = Ks + KV_HALF;
      ++it;
    } else if (nk > 0) {
      KVPool pool;
      pool.base = a.kv + (size_t)st.layer * a.kv_layer_bytes;
      pool.ptab = a.ptab;
      pool.ppr = a.ppr;
      pool.n_heads = a.heads;
      const bf16* ks = kv_ptr<bf16>(pool, slot, k_lo, 0, head);
      const bf16* vs = kv_ptr<bf16>(pool, slot, k_lo, 1, head);
      for (int idx = tid; idx < nk * (WS_DH / 8); idx += NCT) {
        reinterpret_cast<uint4*>(Ks)[idx] = __ldcg(reinterpret_cast<const uint4*>(ks) + idx);
        reinterpret_cast<uint4*>(Vs)[idx] = __ldcg(reinterpret_cast<const uint4*>(vs) + idx);
      }
    }
    // values of keys nk..63 meet a zero weight in P V: make them finite
    for (int idx = nk * (WS_DH / 8) + tid; idx < WS_XCHUNK * (WS_DH / 8); idx += NCT)
      reinterpret_cast<uint4*>(Vs)[idx] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();      // the slot is refilled by TMA after it is released
    compute_sync();
    if (sh.abort) return;
    // ---- the chunk's partial for all rows (one warp, tensor cores)
    if (warp == 0) {
      auto part = [&](int j) {
        return a.apart + ((((size_t)i * H + j) * a.heads + head) * nsplit + sp) * WS_ATTN_PART;
      };
      if (nk > 0) {
        uint32_t qf[4][4];
        attn_q_frags(a.q, a.d, i * H, H, head * WS_DH, qf);
        auto vis = [&](int j) {
          if (j >= H) return 0;
          if (cross) return nk;
          if (j >= nrow) return 0;
          return max(0, min(k_hi, min(Lr + j + 1, a.max_pos)) - k_lo);
        };
        const int g = lane >> 2;
        attn_chunk_partial<false>(Ks, Vs, qf, vis(g), vis(g + 8), H, part);
      } else {
        for (int j = 0; j < H; ++j) {
          float* p = part(j);
          if (lane == 0) { p[0] = -INFINITY; p[1] = 0.f; }
          p[2 + 2 * lane] = 0.f;
          p[3 + 2 * lane] = 0.f;
        }
      }
    }
    if (cross) {
      compute_sync();
      if (tid == 0) mbar_arrive(&sh.empty[s]);
    }
    // ---- the last split of (request, head) folds the partials in split order
    __threadfence();
    compute_sync();
    if (tid == 0) {
      int* c = a.actr + (size_t)i * a.heads + head;
      const int old = atomicAdd(c, 1);
      const int last = old == nsplit - 1;
      if (last) *c = 0;
      sh.flag = last;
    }
    compute_sync();
    if (sh.flag) {
      __threadfence();
      for (int j = warp; j < H; j += NCW) {
        const float* p = a.apart + (((size_t)i * H + j) * a.heads + head) * nsplit * WS_ATTN_PART;
        float o0, o1;
        attn_fold_row<false>(p, nsplit, o0, o1);
        bf16* o = a.ao + ((size_t)i * H + j) * a.d + head * WS_DH + 2 * lane;
        o[0] = __float2bfloat16_rn(o0);
        o[1] = __float2bfloat16_rn(o1);
      }
    }
    compute_sync();      // scratch free for the next unit
  }
}

// ------------------------------------------------------------------ embedding and argmax
// Row r (one per CTA): x = E[token] + P[position]; records where the block
// starts for the drafter history; clears the row's argmax key.
__device__ void embed_stage(const FusedArgs& a) {
  const int r = blockIdx.x, tid = threadIdx.x - 32;
  if (r >= a.M) return;
  int slot, j, pos;
  const bool valid = row_info(a.rm, r, slot, j, pos);
  const int i = r / a.H;
  int tok = a.block[r];
  const bool in_block = j < a.block_len[i];
  if (tid == 0 && in_block && pos >= a.max_pos) atomicOr(a.status, WS_ST_POS);
  if (!valid) { tok = 0; pos = min(pos, a.max_pos - 1); }
  if (tok < 0 || tok >= a.V) {
    if (tid == 0) atomicOr(a.status, WS_ST_TOKEN);
    tok = 0;
  }
  if (tid == 0) {
    if (j == 0) {
      a.pend_start[slot] = a.rm.L[slot];
      a.pend_n[slot] = a.block_len[i];
    }
    a.amax[r] = 0ull;
  }
  const bf16* e = a.tok_emb + (size_t)tok * a.d;
  const bf16* p = a.pos_emb + (size_t)pos * a.d;
  for (int n = tid; n < a.d; n += NCT) a.x[(size_t)r * a.d + n] = __bfloat162float(e[n]) + __bfloat162float(p[n]);
}

__device__ void argmax_stage(const FusedArgs& a) {
  if (blockIdx.x != 0) return;
  for (int r = threadIdx.x - 32; r < a.M; r += NCT) {
    const int i = r / a.H, j = r - i * a.H;
    const bool valid = j < a.block_len[i];
    a.target[(size_t)i * a.H + j] = valid ? argmax_key_id(__ldcg(a.amax + r)) : -1;
  }
}

__device__ void compute(const FusedArgs& a, uint8_t* ring, uint8_t* work, Shared& sh) {
  uint32_t it = 0, done_ph = 0, la_ph = 0;
  int off = 0;
  const int tid = threadIdx.x - 32;
  if (tid < a.M) {
    int slot, j, pos;
    const bool valid = row_info(a.rm, tid, slot, j, pos);
    sh.row_slot[tid] = slot;
    sh.row_j[tid] = j;
    sh.row_pos[tid] = pos;
    sh.row_valid[tid] = valid;
    sh.row_page[tid] = valid ? a.ptab[slot * a.ppr + pos / WS_PAGE] : 0;
  }
  compute_sync();
  for (int g = 0; g < a.n_stages; ++g) {
    const FusedStage& st = a.stages[g];
    const int u0 = first_unit(off);
    off += stage_units(a, st);
    switch (st.kind) {
      case FS_EMBED: embed_stage(a); break;
      case FS_GEMM: gemm_stage(a, st, u0, ring, work, sh, it, done_ph, la_ph); break;
      case FS_SELF:
      case FS_CROSS: attn_stage(a, st, u0, ring, work, sh, it); break;
      default: argmax_stage(a); break;
    }
    compute_sync();
    if (sh.abort) return;
    if (g + 1 < a.n_stages && !grid_sync(a, sh)) return;
  }
}

__global__ void __launch_bounds__(NT, 1) fused_verify_kernel(const __grid_constant__ FusedArgs a) {
  extern __shared__ uint8_t dsm[];
  __shared__ Shared sh;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = base;
  uint8_t* work = base + (size_t)a.ring_slots * SLOT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.ring_slots; ++s) { mbar_init(&sh.full[s], 1); mbar_init(&sh.empty[s], 1); }
    mbar_init(&sh.mma_done, 1);
    mbar_init(&sh.la_bar, 1);
    sh.abort = 0;
    sh.issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&sh.tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    if (lane == 0) producer(a, ring, sh);
    __syncwarp();
  } else {
    compute(a, ring, work, sh);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) drain(a, sh);
  __syncthreads();
  if (warp == 1) tmem_dealloc(sh.tmem_base, TMEM_COLS);
}

constexpr size_t SMEM_LIMIT = 232448;   // 227 KB per CTA (sm_100 family)

size_t dyn_smem(int ring_slots, size_t work_bytes) { return 1024 + (size_t)ring_slots * SLOT + work_bytes; }

}  // namespace

size_t fused_work_bytes(int max_unit_kb) {
  const size_t b = (size_t)max_unit_kb * BKB;
  return b > (size_t)ATT_BYTES ? b : (size_t)ATT_BYTES;
}

int fused_prepare(size_t work_bytes, int* grid_ctas) {
  const size_t stat = sizeof(Shared) + 64;
  if (SMEM_LIMIT < stat + 1024 + work_bytes + 2 * SLOT) return 0;
  int slots = (int)((SMEM_LIMIT - stat - 1024 - work_bytes) / SLOT);
  if (slots > FUSED_MAX_RING) slots = FUSED_MAX_RING;
  const size_t smem = dyn_smem(slots, work_bytes);
  if (cudaFuncSetAttribute(fused_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int coop = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_verify_kernel, NT, smem) != cudaSuccess ||
      per_sm < 1)
    return 0;
  *grid_ctas = sms;
  return slots;
}

cudaError_t launch_fused_verify(const FusedArgs& a, int grid, size_t work_bytes, cudaStream_t s) {
  if (a.M < 1 || a.M > MAXR || a.ring_slots < 2 || a.ring_slots > FUSED_MAX_RING) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = dyn_smem(a.ring_slots, work_bytes);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: the grid barriers need it
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, fused_verify_kernel, a);
}
