// tcgen05 GEMM engine for the bf16 model: Y[token, feature] = X[token, :] . W[feature, :]
//
// Blackwell datapath, written with inline PTX:
//   * TMA (cp.async.bulk.tensor.2d, 128-byte swizzle) streams 128x64 weight
//     tiles and BNx64 activation tiles into a shared-memory ring, completing
//     on mbarriers;
//   * one elected thread issues tcgen05.mma.cta_group::1.kind::f16 (M = 128
//     weight rows, N = BN tokens, K = 16 per instruction) with fp32
//     accumulators in tensor memory (TMEM), and releases each ring slot with
//     tcgen05.commit;
//   * four warps read the accumulator back with tcgen05.ld and run the shared
//     epilogue (bias, GELU, residual, KV-cache scatter, RoPE, logits/argmax).
// Weights are the 128-row A operand ("swap AB"), so a decode step with a
// handful of tokens still fills the MMA M dimension and each token is one
// column: every output element accumulates its k-blocks in the same order
// whatever the number of tokens.  Split-K (fixed per weight shape, never per
// token count) spreads small-M GEMMs over the SMs: the splits of a tile form
// one thread-block cluster whose ranks each add the fp32 partials of their
// share of the token columns in split order through distributed shared
// memory.  A one-token-tile GEMM whose input is the layer norm of the
// residual builds that operand itself.
//
// Each kernel releases its dependents (programmatic dependent launch) right
// after its prologue, and issues the weight TMA loads of the first ring slots
// before griddepcontrol.wait, so the next GEMM's weight stream overlaps the
// current kernel.  Every mbarrier wait is bounded (clock budget); a timeout
// sets a device status bit instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cooperative_groups.h>

#include <mutex>

#include "ws_epilogue.cuh"
#include "ws_tc.cuh"

namespace {

using namespace tc;

struct TcParams {
  int M, N, K;           // tokens, weight rows (features), reduction
  int kb_total;          // K / BK
  int splits;            // split-K factor (grid.x = tiles_f * splits)
  int tiles_f, tiles_t;
  int nz;                // batch entries (CROSSKV: requests)
  int32_t* status;
  // Layer-norm input (split-K, one token tile, all k-blocks of a CTA in the
  // ring at once): B = LayerNorm(ln_x; ln_g, ln_b) built in the kernel, rows
  // of ln_x K floats apart; ln_x == nullptr: B is loaded through tmX.
  const float* ln_x;
  const void* ln_g;
  const void* ln_b;
};

// Fast epilogues: per tile, each thread's feature constants (bias, q/k/v
// part, head, output column) are taken once, then every column is one add
// (and GELU) and one store.  Per element the arithmetic is epi_pair's, so
// results match the generic path bit for bit.  tok[c] (QKV only): element
// offset of token t0 + c's cache row in a K/V page, or -1 where the token is
// not written.  xpre (RESID, optional): the 16 residual values of this
// thread's feature, already loaded.
__device__ __forceinline__ bool fast_epilogue_kind(int kind, const Epi& e) {
  return kind == EPI_STORE || kind == EPI_GELU || kind == EPI_CROSSKV || kind == EPI_QKV ||
         (kind == EPI_RESID && e.hist == nullptr);
}

// Bias of feature n as the fast epilogue adds it (q / v bias for QKV, none for k).
__device__ __forceinline__ float fast_bias(int kind, const Epi& e, int n) {
  if (kind == EPI_QKV || kind == EPI_CROSSKV) {
    const int part = n / e.d, nn = n - part * e.d;
    if (kind == EPI_QKV) return part == 0 ? bias_at<bf16>(e.bias, nn) : part == 2 ? bias_at<bf16>(e.bias2, nn) : 0.0f;
    return part == 1 ? bias_at<bf16>(e.bias2, nn) : 0.0f;
  }
  return bias_at<bf16>(e.bias, n);
}

// Columns c_lo <= c < c_hi of the 16 are stored (the others are another
// CTA's share of a split-K tile).
__device__ __forceinline__ void fast_epilogue16(int kind, const Epi& e, int N, int t, int M, int n, int z, const float* v,
                                                const int* tok, int c0, const float* xpre = nullptr,
                                                const float* bpre = nullptr, int c_lo = 0, int c_hi = 16) {
  if (n >= N) return;
  const int cmax = min(c_hi, M - t);
  switch (kind) {
    case EPI_STORE:
    case EPI_GELU: {
      const float b = bpre ? *bpre : bias_at<bf16>(e.bias, n);
      bf16* o = reinterpret_cast<bf16*>(e.out) + (size_t)t * e.ldo + n;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (c >= c_lo && c < cmax) {
          float y = v[c] + b;
          if (kind == EPI_GELU) y = gelu_erf(y);
          o[(size_t)c * e.ldo] = __float2bfloat16_rn(y);
        }
      }
      break;
    }
    case EPI_RESID: {
      const float b = bpre ? *bpre : bias_at<bf16>(e.bias, n);
      float* x = e.resid + (size_t)t * e.ldr + n;
      float xr[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c >= c_lo && c < cmax) xr[c] = xpre ? xpre[c] : __ldcg(x + (size_t)c * e.ldr);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c >= c_lo && c < cmax) x[(size_t)c * e.ldr] = xr[c] + (v[c] + b);
      break;
    }
    case EPI_CROSSKV: {
      const int part = n / e.d, nn = n - part * e.d;
      const float b = part == 1 ? bias_at<bf16>(e.bias2, nn) : 0.0f;
      bf16* o = xkv_ptr<bf16>(e.xkv, e.req_ids[z], e.xlayer, part, nn / WS_DH, t) + (nn % WS_DH);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c >= c_lo && c < cmax) o[(size_t)c * WS_DH] = __float2bfloat16_rn(part == 1 ? v[c] + b : v[c]);
      break;
    }
    case EPI_QKV: {
      const int part = n / e.d, nn = n - part * e.d;
      if (part == 0) {
        const float b = bpre ? *bpre : bias_at<bf16>(e.bias, nn);
        bf16* o = reinterpret_cast<bf16*>(e.out) + (size_t)t * e.d + nn;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (c >= c_lo && c < cmax) o[(size_t)c * e.d] = __float2bfloat16_rn(v[c] + b);
      } else {
        const float b = bpre ? *bpre : (part == 2 ? bias_at<bf16>(e.bias2, nn) : 0.0f);
        bf16* base = reinterpret_cast<bf16*>(e.kv.base) +
                     ((size_t)(part - 1) * e.kv.n_heads + nn / WS_DH) * (WS_PAGE * WS_DH) + (nn % WS_DH);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (c >= c_lo && c < cmax) {
            const int off = tok[c0 + c];
            if (off >= 0) base[off] = __float2bfloat16_rn(part == 2 ? v[c] + b : v[c]);
          }
        }
      }
      break;
    }
    default:
      break;
  }
}

// KIND >= 0: compiled for that epilogue kind only (the host picks it from
// e.kind); -1: any kind, read from e.kind.
template <int BN, int STAGES, int KIND>
__global__ void __launch_bounds__(128, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, TcParams p,
                   Epi e) {
  const int kind = KIND >= 0 ? KIND : e.kind;
  constexpr int B_BYTES = BN * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  constexpr uint32_t IDESC = idesc_bf16(BM, BN);
  static_assert(BN * BM * 4 <= STAGES * STAGE_BYTES, "a split-K partial must fit in the ring");
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], done;
  __shared__ uint32_t tmem_base;

  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_f = blockIdx.x / p.splits, split = blockIdx.x - tile_f * p.splits;
  const int f0 = tile_f * BM, t0 = blockIdx.y * BN, z = blockIdx.z;
  const int kb0 = (int)((long long)split * p.kb_total / p.splits);
  const int kb1 = (int)((long long)(split + 1) * p.kb_total / p.splits);
  const int nkb = kb1 - kb0;
  // columns of each 16-column group this CTA stores: all, or with split K its
  // share (the cluster rank of a split is its index)
  const int c_lo = p.splits > 1 ? split * 16 / p.splits : 0;
  const int c_hi = p.splits > 1 ? (split + 1) * 16 / p.splits : 16;
  const bool lnin = BN == 16 && p.ln_x != nullptr;
  const uint32_t stage_tx = lnin ? (uint32_t)A_BYTES : (uint32_t)STAGE_BYTES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(&done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(&tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // Let the next kernel launch now: its prologue and weight prefetch overlap
  // this kernel (it still waits for our completion before reading outputs).
  pdl_trigger();

  // Row count: a host value, except for the acoustic K/V GEMM whose per-request
  // frame ranges live in device memory (read only after the dependency wait).
  int M = p.M, row0 = 0;
  const bool early = kind != EPI_CROSSKV;
  if (!early) {
    pdl_wait();
    row0 = e.cu_frames[z];
    M = min(e.cu_frames[z + 1] - row0, e.xkv.max_frames);
  }
  const bool active = t0 < M && nkb > 0;
  // ---- weights of the first ring slots: independent of the previous kernel
  const int npre = active ? (nkb < STAGES ? nkb : STAGES) : 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < npre; ++i) {
      mbar_expect_tx(&full[i], stage_tx);
      tma_load_2d(ring + i * STAGE_BYTES, &tmW, &full[i], (kb0 + i) * BK, f0);
    }
  }
  // layer-norm gain and bias of this CTA's k-range are weights: into shared
  // memory now (16 bytes a thread), read after the dependency wait
  __shared__ __align__(16) bf16 ln_gb[2][STAGES * BK];
  if (lnin && active && (int)threadIdx.x < nkb * 16) {
    const int h = threadIdx.x >> 3 & 1, off = (threadIdx.x >> 4) * BK + (threadIdx.x & 7) * 8;
    const bf16* src = reinterpret_cast<const bf16*>(h ? p.ln_b : p.ln_g) + kb0 * BK + off;
    *reinterpret_cast<uint4*>(&ln_gb[h][off]) = *reinterpret_cast<const uint4*>(src);
  }
  // the bias of this thread's feature is a weight: load it before the wait
  float bpre = 0.0f;
  if (BN == 16 && active && (kind == EPI_RESID || kind == EPI_QKV || kind == EPI_STORE || kind == EPI_GELU) &&
      f0 + warp * 32 + lane < p.N)
    bpre = fast_bias(kind, e, f0 + warp * 32 + lane);
  // Cache rows of the tile's tokens (QKV): positions, request slots and the
  // page table were all written before this library call began, so the
  // table is built before the dependency wait.
  __shared__ int tok_tab[16];
  if (BN == 16 && active && kind == EPI_QKV && threadIdx.x < 16) {
    int slot, j, pos, off = -1;
    const int r = t0 + (int)threadIdx.x;
    if (r < M && row_info(e.rm, r, slot, j, pos)) {
      const int page = e.kv.ptab[slot * e.kv.ppr + pos / WS_PAGE];
      off = (int)((size_t)page * 2 * e.kv.n_heads * (WS_PAGE * WS_DH) + (size_t)(pos % WS_PAGE) * WS_DH);
    }
    tok_tab[threadIdx.x] = off;
  }
  if (early) pdl_wait();

  // Epilogue inputs that do not depend on the MMAs are loaded now, while the
  // weights stream (one-token-tile calls): this thread's residual values.
  float xpre[16];
  const bool pre_resid = BN == 16 && active && kind == EPI_RESID && e.hist == nullptr;
  if (pre_resid) {
    const int pn = f0 + warp * 32 + lane;
#pragma unroll
    for (int c = 0; c < 16; ++c)
      xpre[c] = (c >= c_lo && c < c_hi && t0 + c < M && pn < p.N) ? __ldcg(e.resid + (size_t)(t0 + c) * e.ldr + pn)
                                                                  : 0.0f;
  }
  const bool fast16 = BN == 16 && (pre_resid || kind == EPI_QKV || kind == EPI_STORE || kind == EPI_GELU);

  if (lnin && active) {
    // B = LayerNorm(x) for token rows t0 .. t0 + 15 and this CTA's k-blocks,
    // written into the B half of ring slot i (k-block kb0 + i) in the layout a
    // 16-row x 64-column TMA box with 128-byte swizzle has: row r at byte
    // r * 128, 16-byte chunk c at chunk c ^ (r & 7).  Warp w normalises rows
    // w, w + 4, w + 8, w + 12 (all loads of a warp in one memory round trip)
    // with the layer-norm kernel's per-row warp arithmetic, so the operand is
    // bit-identical to the normalised copy that kernel would write.
    const int nr = min(BN, M - t0), k_lo = kb0 * BK;
    const int nrw = nr > warp ? (nr - warp + 3) >> 2 : 0;     // rows warp + 4j < nr
    const float* xs[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) xs[j] = p.ln_x + (size_t)(t0 + warp + 4 * j) * p.K;   // read for j < nrw only
    __syncthreads();                   // gain and bias staged
    ln_rows_warp<true, 4, 10>(
        xs, nrw, p.K, ln_gb[0], ln_gb[1], true,
        [&](int j, int k, float v0, float v1, float v2, float v3) {
          const int r = warp + 4 * j, kl = k - k_lo, col = kl & 63;
          __nv_bfloat162 h0 = __floats2bfloat162_rn(v0, v1), h1 = __floats2bfloat162_rn(v2, v3);
          uint2 w;
          w.x = *reinterpret_cast<uint32_t*>(&h0);
          w.y = *reinterpret_cast<uint32_t*>(&h1);
          *reinterpret_cast<uint2*>(ring + (kl >> 6) * STAGE_BYTES + A_BYTES + r * 128 +
                                    ((((col >> 3) ^ (r & 7)) << 4) | ((col & 7) * 2))) = w;
        },
        k_lo, kb1 * BK, k_lo);
    for (int idx = threadIdx.x; idx < (BN - nr) * nkb * 8; idx += 128) {   // rows nr .. 15 are zero
      const int r = nr + idx / (nkb * 8), rem = idx % (nkb * 8);
      *reinterpret_cast<uint4*>(ring + (rem >> 3) * STAGE_BYTES + A_BYTES + r * 128 + ((rem & 7) << 4)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor core
    __syncthreads();
  }

  if (threadIdx.x == 0 && active) {
    // ---- producer
    if (!lnin)
      for (int i = 0; i < npre; ++i)
        tma_load_2d(ring + i * STAGE_BYTES + A_BYTES, &tmX, &full[i], (kb0 + i) * BK, row0 + t0);
    for (int i = npre; i < nkb; ++i) {     // (none with a layer-norm input: nkb <= STAGES)
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)((i / STAGES) & 1);
      if (!mbar_wait(&empty[s], ph ^ 1u)) { atomicOr(p.status, WS_ST_TIMEOUT); break; }
      mbar_expect_tx(&full[s], STAGE_BYTES);
      uint8_t* st = ring + s * STAGE_BYTES;
      tma_load_2d(st, &tmW, &full[s], (kb0 + i) * BK, f0);
      tma_load_2d(st + A_BYTES, &tmX, &full[s], (kb0 + i) * BK, row0 + t0);
    }
  }
  if (warp == 1 && lane == 0 && active) {
    // ---- MMA issuer
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)((i / STAGES) & 1);
      if (!mbar_wait(&full[s], ph)) { atomicOr(p.status, WS_ST_TIMEOUT); break; }
      tc_fence_after();
      const uint32_t a = smem_u32(ring + s * STAGE_BYTES), b = a + A_BYTES;
      const uint64_t ad = sdesc_sw128(a), bd = sdesc_sw128(b);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        umma_bf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), IDESC, (i | kk) != 0 ? 1u : 0u);
      umma_commit(&empty[s]);
    }
    umma_commit(&done);
  }
  __syncwarp();

  bool ok = true;
  if (active) {
    ok = mbar_wait(&done, 0);
    if (!ok) atomicOr(p.status, 8);
  }
  ok = __syncthreads_and(ok) != 0;      // CTA-uniform before any further barrier
  tc_fence_after();

  const int row = warp * 32 + lane;            // TMEM lane == weight row of the tile
  const int n = f0 + row;
  const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
  // Split-K: the splits of one tile form a thread-block cluster.  Each CTA
  // parks its fp32 partial in its own (now idle) ring memory; after a
  // cluster barrier every rank folds its own share of each 16-column group
  // (columns [c_lo, c_hi)), reading the partials of ranks 0, 1, 2, ...
  // through distributed shared memory and adding them in that order, and
  // stores those columns; the ranks' shares are disjoint and cover the
  // group.  Every CTA of an active cluster reaches both cluster barriers,
  // also after a timed-out wait.  One epilogue call site serves both paths
  // (the code stays small: a layer's projections all run this kernel).
  namespace cg = cooperative_groups;
  const bool splitk = p.splits > 1;
  float* mine = reinterpret_cast<float*>(ring);
  if (active && splitk) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      float v[16];
      if (ok) tmem_ld16(taddr + (uint32_t)c0, v);
#pragma unroll
      for (int c = 0; c < 16; ++c) mine[(c0 + c) * BM + row] = ok ? v[c] : 0.0f;
    }
    cg::this_cluster().sync();
  }
  if (active && (splitk || ok)) {
    const float* part[8];
    if (splitk) {
      cg::cluster_group cl = cg::this_cluster();
#pragma unroll
      for (int r = 0; r < 8; ++r) part[r] = cl.map_shared_rank(mine, r < p.splits ? r : 0);
    }
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      float v[16];
      if (splitk) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float a = 0.0f;
          if (c >= c_lo && c < c_hi) {
            a = part[0][(c0 + c) * BM + row];
#pragma unroll
            for (int r = 1; r < 8; ++r)
              if (r < p.splits) a += part[r][(c0 + c) * BM + row];
          }
          v[c] = a;
        }
        // the last group's reads of the others' partials are done: arrive
        // now, and wait (for the others' reads of this CTA's partial) only
        // before exit, so the barrier's latency overlaps the stores
        if (c0 + 16 >= BN) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
      } else {
        tmem_ld16(taddr + (uint32_t)c0, v);
      }
      if (fast16) fast_epilogue16(kind, e, p.N, t0 + c0, M, n, z, v, tok_tab, c0, pre_resid ? xpre : nullptr, &bpre,
                                  splitk ? c_lo : 0, splitk ? c_hi : 16);
      else epi_columns16(kind, e, p.N, t0 + c0, n, M, z, v, splitk ? c_lo : 0, splitk ? c_hi : 16);
    }
    if (splitk) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ persistent variant
// Calls without split-K (all large-token GEMMs, the acoustic K/V projection,
// the LM head) run as a persistent, warp-specialised kernel: one CTA per SM
// walks tiles t = blockIdx.x, + gridDim.x, ... (feature tile fastest, so
// the CTAs of a wave share the activation tile in L2).  Warp 0 streams
// weight and activation tiles through the ring, warp 1 issues the MMAs into
// one of two TMEM accumulators, warps 2..9 run the epilogue of tile i while
// the MMAs of tile i+1 proceed: two warps per TMEM lane quarter (a warp may
// only read its own quarter), each taking alternate 16-column groups, so the
// bias / GELU / residual arithmetic of a wide tile keeps pace with its MMAs.  A tile's k
// order is that of gemm_tc_kernel, so both give bit-identical outputs.
template <int BN>
constexpr int persistent_stages() { return (200 * 1024) / (A_BYTES + BN * BK * 2); }

template <int BN>
constexpr int persistent_smem() { return persistent_stages<BN>() * (A_BYTES + BN * BK * 2) + 1024; }

struct TileInfo { int tile_f, t0, z, row0, M; bool active; };

__device__ __forceinline__ TileInfo tile_of(const TcParams& p, const Epi& e, int kind, int t, int BN) {
  TileInfo ti;
  ti.tile_f = t % p.tiles_f;
  const int rest = t / p.tiles_f;
  const int tt = rest % p.tiles_t;
  ti.z = rest / p.tiles_t;
  ti.t0 = tt * BN;
  ti.row0 = 0;
  ti.M = p.M;
  if (kind == EPI_CROSSKV) {        // per-request frame ranges (device memory, read after the dependency wait)
    ti.row0 = e.cu_frames[ti.z];
    ti.M = min(e.cu_frames[ti.z + 1] - ti.row0, e.xkv.max_frames);
  }
  ti.active = ti.t0 < ti.M;
  return ti;
}

constexpr int PERSIST_THREADS = 320;        // producer, MMA issuer, 8 epilogue warps

template <int BN, int KIND>
__global__ void __launch_bounds__(PERSIST_THREADS, 1)
    gemm_tc_persistent(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, TcParams p,
                       Epi e) {
  const int kind = KIND >= 0 ? KIND : e.kind;
  constexpr int STAGES = persistent_stages<BN>();
  constexpr int B_BYTES = BN * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t ACC_COLS = BN < 32 ? 32 : BN;
  constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
  constexpr uint32_t IDESC = idesc_bf16(BM, BN);
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base, issued;
  __shared__ int tok_tab[BN];

  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.tiles_f * p.tiles_t * p.nz;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], 8); }
    issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(&tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer.  Weights of the first tile's first slots go out before
      // the dependency wait (they do not depend on the previous kernel).
      int npre = 0;
      if (kind != EPI_CROSSKV && blockIdx.x < T) {
        const TileInfo ti = tile_of(p, e, kind, blockIdx.x, BN);
        if (ti.active) {
          npre = p.kb_total < STAGES ? p.kb_total : STAGES;
          for (int i = 0; i < npre; ++i) {
            mbar_expect_tx(&full[i], STAGE_BYTES);
            tma_load_2d(ring + i * STAGE_BYTES, &tmW, &full[i], i * BK, ti.tile_f * BM);
          }
        }
      }
      pdl_wait();
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
        const TileInfo ti = tile_of(p, e, kind, t, BN);
        if (!ti.active) continue;
        for (int kb = 0; kb < p.kb_total; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          uint8_t* st = ring + s * STAGE_BYTES;
          if ((int)it >= npre) {
            if (!mbar_wait(&empty[s], ((it / STAGES) & 1u) ^ 1u)) { atomicOr(p.status, WS_ST_TIMEOUT); ok = false; break; }
            mbar_expect_tx(&full[s], STAGE_BYTES);
            tma_load_2d(st, &tmW, &full[s], kb * BK, ti.tile_f * BM);
          }
          tma_load_2d(st + A_BYTES, &tmX, &full[s], kb * BK, ti.row0 + ti.t0);
        }
      }
      issued = it > (uint32_t)npre ? it : (uint32_t)npre;
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
        if (kind == EPI_CROSSKV && t == (int)blockIdx.x) pdl_wait();
        const TileInfo ti = tile_of(p, e, kind, t, BN);
        if (!ti.active) continue;
        const uint32_t acc = local & 1u;
        if (!mbar_wait(&acc_empty[acc], ((local >> 1) & 1u) ^ 1u)) { atomicOr(p.status, WS_ST_TIMEOUT); break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * ACC_COLS;
        for (int kb = 0; kb < p.kb_total; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          if (!mbar_wait(&full[s], (it / STAGES) & 1u)) { atomicOr(p.status, WS_ST_TIMEOUT); ok = false; break; }
          tc_fence_after();
          const uint32_t a = smem_u32(ring + s * STAGE_BYTES), b = a + A_BYTES;
          const uint64_t ad = sdesc_sw128(a), bd = sdesc_sw128(b);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), IDESC, (kb | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        umma_commit(&acc_full[acc]);
        ++local;
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: warps 2..9; warp w reads TMEM lane quarter w % 4 and
    // the column groups 16 h, 16 h + 32, ... with h = (w - 2) / 4
    pdl_wait();
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const bool fast = fast_epilogue_kind(kind, e);
    uint32_t local = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      const TileInfo ti = tile_of(p, e, kind, t, BN);
      if (!ti.active) continue;
      if (kind == EPI_QKV) {
        // cache rows of this tile's tokens (one entry per column)
        asm volatile("bar.sync 1, 256;" ::: "memory");
        for (int c = row + half * 128; c < BN; c += 256) {
          int slot, j, pos, off = -1;
          const int r = ti.t0 + c;
          if (r < ti.M && row_info(e.rm, r, slot, j, pos)) {
            const int page = e.kv.ptab[slot * e.kv.ppr + pos / WS_PAGE];
            off = (int)((size_t)page * 2 * e.kv.n_heads * (WS_PAGE * WS_DH) + (size_t)(pos % WS_PAGE) * WS_DH);
          }
          tok_tab[c] = off;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
      }
      const int n = ti.tile_f * BM + row;
      // Residual epilogue on tiles of 64 or 128 tokens: the residual values
      // of this warp's column groups do not depend on the MMAs, so they are
      // read before the accumulator wait instead of one round trip per group
      // after it (the stores of a group would otherwise hold back the next
      // group's loads: both address the residual rows).
      constexpr bool PRE = KIND == EPI_RESID && BN >= 64 && BN <= 128;
      constexpr int NPG = PRE ? BN / 32 : 1;
      float xpre[NPG][16];
      if (PRE) {
#pragma unroll
        for (int q = 0; q < NPG; ++q)
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int r = ti.t0 + half * 16 + 32 * q + c;
            xpre[q][c] = (r < ti.M && n < p.N) ? __ldcg(e.resid + (size_t)r * e.ldr + n) : 0.0f;
          }
      }
      const uint32_t acc = local & 1u;
      const bool ok = mbar_wait(&acc_full[acc], (local >> 1) & 1u);
      if (!ok) { if (lane == 0) atomicOr(p.status, WS_ST_TIMEOUT); break; }
      tc_fence_after();
      const uint32_t taddr = tmem + acc * ACC_COLS + ((uint32_t)(quarter * 32) << 16);
      if constexpr (PRE) {
#pragma unroll
        for (int q = 0; q < NPG; ++q) {
          const int c0 = half * 16 + 32 * q;
          if (ti.t0 + c0 >= ti.M) break;
          float v[16];
          tmem_ld16(taddr + (uint32_t)c0, v);
          fast_epilogue16(kind, e, p.N, ti.t0 + c0, ti.M, n, ti.z, v, tok_tab, c0, xpre[q]);
        }
      } else {
#pragma unroll 1
        for (int c0 = half * 16; c0 < BN; c0 += 32) {
          if (ti.t0 + c0 >= ti.M) break;
          float v[16];
          tmem_ld16(taddr + (uint32_t)c0, v);
          if (fast) fast_epilogue16(kind, e, p.N, ti.t0 + c0, ti.M, n, ti.z, v, tok_tab, c0);
          else epi_columns16(kind, e, p.N, ti.t0 + c0, n, ti.M, ti.z, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&acc_empty[acc])) : "memory");
      ++local;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    // every copy issued has landed (bounded), also after an early stop
    const uint32_t n = issued, first = n > (uint32_t)STAGES ? n - STAGES : 0u;
    for (uint32_t it = first; it < n; ++it)
      if (!mbar_wait(&full[it % STAGES], (it / STAGES) & 1u)) { atomicOr(p.status, WS_ST_TIMEOUT); break; }
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

int g_sm_count = 0;

// The instance for e's epilogue kind: specialised for the kinds of the
// decoder's batch-1 LM head and the encoder's projections, else generic.
template <int BN>
auto persistent_for(const Epi& e) -> decltype(&gemm_tc_persistent<BN, -1>) {
  if constexpr (BN == 16) {
    if (e.kind == EPI_LOGITS) return gemm_tc_persistent<BN, EPI_LOGITS>;
  }
  if constexpr (BN >= 64) {
    if (e.kind == EPI_STORE) return gemm_tc_persistent<BN, EPI_STORE>;
    if (e.kind == EPI_GELU) return gemm_tc_persistent<BN, EPI_GELU>;
    if (e.kind == EPI_RESID && e.hist == nullptr) return gemm_tc_persistent<BN, EPI_RESID>;
  }
  return gemm_tc_persistent<BN, -1>;
}

template <int BN>
cudaError_t launch_persistent(const GemmShape& g, const Epi& e, const CUtensorMap& mw, const CUtensorMap& mx,
                              const TcParams& p, cudaStream_t s, bool pdl) {
  const int T = p.tiles_f * p.tiles_t * p.nz;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g_sm_count > 0 && T > g_sm_count ? g_sm_count : T);
  cfg.blockDim = dim3(PERSIST_THREADS);
  cfg.dynamicSmemBytes = persistent_smem<BN>();
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, persistent_for<BN>(e), mw, mx, p, e);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

template <int BN, int STAGES>
constexpr int tc_smem() {
  return STAGES * (A_BYTES + BN * BK * 2) + 1024;
}

template <int BN, int STAGES>
cudaError_t launch_bn(const GemmShape& g, const Epi& e, const CUtensorMap& mw, const CUtensorMap& mx,
                      const TcParams& p, cudaStream_t s, bool pdl) {
  constexpr int smem = tc_smem<BN, STAGES>();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.tiles_f * p.splits, p.tiles_t, g.batch > 0 ? g.batch : 1);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (pdl) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.splits > 1) {      // the splits of a tile are one cluster
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = p.splits;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  ws_count_launches(1);
  // One instance serves every epilogue kind: the decoder's projections of a
  // layer alternate kinds, and a single code body they share stays in the
  // instruction caches (one instance per kind measured slower at batch 1).
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, STAGES, -1>, mw, mx, p, e);
}

}  // namespace

bool tc_engine_available() {
  std::call_once(g_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Row-major bf16 matrix [rows, cols] as a TMA tensor map with 64-column x
// box_rows boxes and 128-byte swizzle.  Returns false when the encoder
// rejects it (alignment, sizes).
bool tc_encode_map(TcMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  if (!tc_engine_available()) return false;
  static_assert(sizeof(TcMap) >= sizeof(CUtensorMap), "TcMap too small");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(reinterpret_cast<CUtensorMap*>(m), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major fp32 matrix [rows, cols] (cols a multiple of 256) as a 3-D TMA
// map {256, cols / 256, rows} whose box holds box_rows whole rows, stored
// row after row in shared memory (no swizzle).  Rows beyond `rows` read as 0.
bool tc_encode_rows_f32(TcMap* m, const float* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  if (!tc_engine_available() || cols % 256 != 0) return false;
  cuuint64_t dims[3] = {256, (cuuint64_t)cols / 256, (cuuint64_t)rows};
  cuuint64_t strides[2] = {256 * 4, (cuuint64_t)cols * 4};
  cuuint32_t box[3] = {256, (cuuint32_t)(cols / 256), box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(reinterpret_cast<CUtensorMap*>(m), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                        const_cast<float*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
template <int BN>
const void* persistent_instance(int k) {
  switch (k) {
    case EPI_STORE: return (const void*)gemm_tc_persistent<BN, EPI_STORE>;
    case EPI_GELU: return (const void*)gemm_tc_persistent<BN, EPI_GELU>;
    case EPI_RESID: return (const void*)gemm_tc_persistent<BN, EPI_RESID>;
    default: return (const void*)gemm_tc_persistent<BN, -1>;
  }
}
}  // namespace

// Raise the dynamic shared-memory limit of every kernel variant once, before
// any launch (so no attribute call happens while a stream is being captured).
cudaError_t tc_init_attributes() {
  cudaError_t r = cudaSuccess;
  auto set = [&](const void* fn, int bytes) {
    if (r == cudaSuccess) r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  };
  set((const void*)gemm_tc_kernel<16, 5, -1>, tc_smem<16, 5>());
  set((const void*)gemm_tc_kernel<32, 5, -1>, tc_smem<32, 5>());
  set((const void*)gemm_tc_kernel<64, 4, -1>, tc_smem<64, 4>());
  set((const void*)gemm_tc_persistent<16, -1>, persistent_smem<16>());
  set((const void*)gemm_tc_persistent<16, EPI_LOGITS>, persistent_smem<16>());
  set((const void*)gemm_tc_persistent<32, -1>, persistent_smem<32>());
  for (int k : {-1, (int)EPI_STORE, (int)EPI_GELU, (int)EPI_RESID}) {
    set(persistent_instance<64>(k), persistent_smem<64>());
    set(persistent_instance<128>(k), persistent_smem<128>());
    set(persistent_instance<256>(k), persistent_smem<256>());
  }
  if (r == cudaSuccess) {
    int dev = 0;
    r = cudaGetDevice(&dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&g_sm_count, cudaDevAttrMultiProcessorCount, dev);
  }
  return r;
}

int tc_bn_index(int bn) { return bn <= 16 ? 0 : bn <= 32 ? 1 : bn <= 64 ? 2 : bn <= 128 ? 3 : 4; }

// Token-tile width.  Up to 64 tokens: the smallest tile that holds them.
// Beyond: the widest of 256 / 128 / 64 whose tile count (feature tiles x
// token tiles x batch) still fills about the SMs.  A row's k order does not
// depend on the width, so the choice never changes a result.
int tc_pick_bn(int M, int N, int batch) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  const int tf = (N + BM - 1) / BM, b = batch > 0 ? batch : 1;
  const int want = g_sm_count > 0 ? g_sm_count * 9 / 10 : 133;
  for (int bn = 256; bn >= 128; bn /= 2)
    if (tf * ((M + bn - 1) / bn) * b >= want) return bn;
  return M <= 128 ? 128 : 64;
}

bool tc_ln_input_ok(int M, int N, int K, int splits) {
  if (M <= 0 || K % 128 != 0 || K > 1280 || tc_pick_bn(M, N, 1) != 16) return false;
  const int kb = K / BK, s = splits < 1 ? 1 : (splits > kb ? kb : splits);
  return s > 1 && (kb + s - 1) / s <= 5;     // 5: ring slots of gemm_tc_kernel<16, 5>
}

cudaError_t launch_gemm_tc(const GemmShape& g, const Epi& e, const TcMap& mw, const TcMap* mx_cached,
                           const void* x_base, uint64_t x_rows, int splits, cudaStream_t s,
                           bool pdl) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  if (g.K % BK != 0 || g.ldx != g.K) return cudaErrorInvalidValue;
  const int BN = tc_pick_bn(g.M, g.N, g.batch);
  TcMap mx;
  if (mx_cached) mx = *mx_cached;
  else if (!tc_encode_map(&mx, x_base, x_rows, (uint64_t)g.K, (uint32_t)BN)) return cudaErrorInvalidValue;
  TcParams p = {};
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.kb_total = g.K / BK;
  p.splits = splits < 1 ? 1 : (splits > p.kb_total ? p.kb_total : splits);
  p.tiles_f = (g.N + BM - 1) / BM;
  p.tiles_t = (g.M + BN - 1) / BN;
  p.nz = g.batch > 0 ? g.batch : 1;
  p.status = e.status;
  // split-K partials live in the ring of each CTA of the cluster: BN <= 64 tokens
  if (p.splits > 1 && BN > 64) p.splits = 1;
  if (g.ln_x) {
    if (g.batch > 1 || !tc_ln_input_ok(g.M, g.N, g.K, p.splits) || !g.ln_g || !g.ln_b) return cudaErrorInvalidValue;
    p.ln_x = g.ln_x; p.ln_g = g.ln_g; p.ln_b = g.ln_b;
  }
  const CUtensorMap& W = *reinterpret_cast<const CUtensorMap*>(&mw);
  const CUtensorMap& X = *reinterpret_cast<const CUtensorMap*>(&mx);
  // Token tiles wider than 64 never split K: they always run persistent, so
  // the split-K kernel is compiled for 16 / 32 / 64 tokens only.
  if (BN > 64 || (p.splits == 1 && g_sm_count > 0)) {
    switch (BN) {
      case 16: return launch_persistent<16>(g, e, W, X, p, s, pdl);
      case 32: return launch_persistent<32>(g, e, W, X, p, s, pdl);
      case 64: return launch_persistent<64>(g, e, W, X, p, s, pdl);
      case 128: return launch_persistent<128>(g, e, W, X, p, s, pdl);
      default: return launch_persistent<256>(g, e, W, X, p, s, pdl);
    }
  }
  switch (BN) {
    case 16: return launch_bn<16, 5>(g, e, W, X, p, s, pdl);
    case 32: return launch_bn<32, 5>(g, e, W, X, p, s, pdl);
    default: return launch_bn<64, 4>(g, e, W, X, p, s, pdl);
  }
}
