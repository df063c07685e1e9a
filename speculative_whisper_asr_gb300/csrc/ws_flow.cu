// Dataflow block verification for one-request contexts (the batch-1 decode
// of Whisper-Flash §3.1: the target scores the anchor and the K proposals in
// one decoder pass).  One cooperative kernel runs the whole target pass:
// token + position embedding, every decoder layer, final layer norm, tied
// LM head and argmax.
//
// Why one kernel, and why no grid barriers: a batch-1 verify reads ~1.6 GB of
// weights but each step is a few KB of activations, and a chain of ~8
// dependent steps per layer.  Kernel-per-step pays a launch and a drain per
// step; a grid barrier per step makes every SM wait for the slowest.  Here
// each step is cut into tasks, every CTA takes one contiguous share of each
// step, and a CTA waits only for the counters of the tasks whose outputs it
// reads:
//   * QKV / cross-query tiles signal per attention head, so a head's
//     attention starts when its 12 (or 4) tiles are stored;
//   * FC2 work on FFN slice s waits only for FC1 slice s;
//   * the output projections wait for all heads, layer norms for the whole
//     residual row (that is what the arithmetic needs).
// Weight streaming does not wait for any of it: warp 0 of each CTA walks the
// CTA's tasks and issues TMA loads of every weight tile (and acoustic K/V
// chunk) into a 16-slot shared-memory ring as soon as a slot is free, so HBM
// reads run ahead across steps and layers.
//
// Tasks.  A projection tile is 16 output features x one d-wide slice of the
// reduction (FC2's 4d reduction is cut into d-wide slices, folded in slice
// order by the last-arriving slice of the tile).  A CTA's tiles of one step
// (a bundle of up to 3 sharing one B operand) are multiplied together: each
// of the four compute warps takes every fourth 64-wide k-block of every tile
// with mma.sync m16n8k16 (bf16 in, fp32 accumulate; weights as A, the <= 16
// block rows as the N = 16 tile), the four partial tiles are added in warp
// order, and warp t runs the fused epilogue of tile t (bias, residual, GELU,
// K/V cache scatter, logits and argmax keys).  At <= 16 rows a projection is
// a weight-streaming GEMV, so the warp-level MMA is the right tool; the
// tcgen05 engine runs the large-batch GEMMs.  Layer-norm inputs come in by
// one TMA box of whole fp32 residual rows and are normalised from shared
// memory.  Attention reuses the tensor-core chunk partial and the fold of the
// per-op kernels: self-attention of a head in one CTA (its chunks on four
// warps, folded in shared memory), cross-attention in groups of four 64-frame
// chunks per CTA (folded in the CTA, then the groups folded by the head's
// last-arriving group).
//
// Every output element's reduction order is fixed by the task layout and
// never depends on the number of block rows, so block verification and
// one-token decoding give bit-identical rows.  Every wait is bounded: a
// timeout sets the device status word and a global abort flag, after which
// every CTA runs out its program without waiting and exits; the last CTA to
// exit zeroes the counters for the next launch.
#include <cuda.h>

#include "ws_attn_common.cuh"
#include "ws_attn_mma.cuh"
#include "ws_flow.cuh"
#include "ws_tc.cuh"

namespace {

using namespace tc;

constexpr int NT = 160;               // warp 0 streams; warps 1..4 compute
constexpr int NCT = 128;              // compute threads
constexpr int NSLOT = 16;             // ring slots
constexpr int SLOT = 8192;            // four k-blocks of a 16-row weight tile, or one K / V chunk
constexpr int KB = 2048;              // 16 rows x 64 bf16: one k-block of a weight or B tile
constexpr int BSM = 40960;            // B operand [d/64][16][64] bf16, or self-attention partials
constexpr int XS = FLOW_XS_BYTES;     // residual rows for a layer norm; reduction / partial scratch
constexpr int GBS = 2 * 1280 * 2;     // layer-norm gain and bias (bf16, d <= 1280)
constexpr int MAXB = 3;               // tiles per bundle (3 x 5 slots <= NSLOT)
constexpr int KVBOX = WS_XCHUNK * WS_DH * 2;   // one 64 x 64 bf16 chunk of K or V
constexpr long long SPIN = 1ll << 31; // clock cycles (~1 s) before a wait gives up

enum Kind { K_EMBED, K_QKV, K_SELF, K_O, K_QC, K_CROSS, K_OC, K_FC1, K_FC2, K_HEAD };

struct Smem {
  uint64_t full[NSLOT], empty[NSLOT], bbar, xbar;
  unsigned long long skey[FLOW_MAX_ROWS];
  uint32_t issued;                     // ring slots the producer armed
  int flag;
  int abort;
  int b_pending, x_pending;            // a B-operand / residual copy may still be in flight ...
  uint32_t b_parity, x_parity;         // ... completing this phase parity of its barrier
};

// Per-call quantities every thread derives the same way at kernel start.
struct Plan {
  int slot, L, blen, Fv;
  int nch_self, nch_x, ngrp;
  int spt;                            // ring slots per tile (d / 256)
  int kbt;                            // k-blocks of a d-wide slice (d / 64)
  int ksplit;                         // FC2 slices (f / d)
};

// ------------------------------------------------------------------ synchronisation helpers
__device__ __forceinline__ int ld_acq(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel(int* p, int v) {
  int r;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(r) : "l"(p), "r"(v) : "memory");
  return r;
}
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ int* gctr(const FlowArgs& a, int i) {
  return a.ctr + (size_t)a.n_layers * FLOW_CTR_LAYER + i;
}
__device__ __forceinline__ int* lctr(const FlowArgs& a, int l, int i) {
  return a.ctr + (size_t)l * FLOW_CTR_LAYER + i;
}

__device__ __forceinline__ void set_abort(const FlowArgs& a, Smem& sh) {
  atomicOr(a.status, WS_ST_TIMEOUT);
  atomicExch(gctr(a, FG_ABORT), 1);
  sh.abort = 1;
}
__device__ __forceinline__ bool aborted(const FlowArgs& a, Smem& sh) {
  if (sh.abort) return true;
  if (*reinterpret_cast<volatile const int*>(gctr(a, FG_ABORT))) { sh.abort = 1; return true; }
  return false;
}

// One thread: wait until *p >= target (acquire).  False on timeout or abort.
__device__ __noinline__ bool wait_ge(const FlowArgs& a, Smem& sh, const int* p, int target) {
  if (sh.abort) return false;
  if (ld_acq(p) >= target) return true;
  const long long t0 = clock64();
  for (;;) {
    if (ld_acq(p) >= target) return true;
    if (aborted(a, sh)) return false;
    if (clock64() - t0 > SPIN) { set_abort(a, sh); return false; }
  }
}

// mbarrier phase wait, bounded, giving up early once the call is aborted.
__device__ __noinline__ bool ring_wait_slow(const FlowArgs& a, Smem& sh, uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  for (int n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (aborted(a, sh)) return false;
      if (clock64() - t0 > SPIN) { set_abort(a, sh); return false; }
    }
  }
}
__device__ __forceinline__ bool ring_wait(const FlowArgs& a, Smem& sh, uint64_t* bar, uint32_t parity) {
  return mbar_try_wait(bar, parity) || ring_wait_slow(a, sh, bar, parity);
}

// ------------------------------------------------------------------ the static schedule
// Every step's units are dealt to the CTAs in contiguous shares, starting
// where the previous step stopped (so small steps land on different SMs):
// with n >= G units CTA r (counted from the step's first CTA) gets units
// [r n / G, (r + 1) n / G), else unit r.
template <class F>
__device__ __forceinline__ void walk(const FlowArgs& a, const Plan& P, F&& f) {
  const int G = gridDim.x, b = blockIdx.x;
  const int dt = a.d / 16;
  const int n_steps = 2 + 8 * a.n_layers;       // embedding, 8 steps per layer, LM head
  int off = 0;
#pragma unroll 1
  for (int i = 0; i < n_steps; ++i) {
    int kind, layer, n;
    if (i == 0) { kind = K_EMBED; layer = 0; n = dt; }
    else if (i == n_steps - 1) { kind = K_HEAD; layer = a.n_layers; n = (a.V + 15) / 16; }
    else {
      layer = (i - 1) >> 3;
      kind = K_QKV + ((i - 1) & 7);
      switch (kind) {
        case K_QKV: n = 3 * dt; break;
        case K_SELF: n = a.heads; break;
        case K_CROSS: n = a.heads * P.ngrp; break;
        case K_FC1: n = a.f / 16; break;
        case K_FC2: n = dt * P.ksplit; break;
        default: n = dt; break;                 // O, QC, OC
      }
    }
    const int r = (b - off % G + G) % G;
    int s0, s1;
    if (n >= G) {
      s0 = (int)((long long)r * n / G);
      s1 = (int)((long long)(r + 1) * n / G);
    } else {
      s0 = r < n ? r : n;
      s1 = r < n ? r + 1 : n;
    }
    if (s1 > s0) f(kind, layer, s0, s1);
    off += min(n, G);
  }
}

__device__ __forceinline__ bool is_weight(int kind) {
  return kind == K_QKV || kind == K_O || kind == K_QC || kind == K_OC || kind == K_FC1 || kind == K_FC2 ||
         kind == K_HEAD;
}
__device__ __forceinline__ bool ln_input(int kind) {
  return kind == K_QKV || kind == K_QC || kind == K_FC1 || kind == K_HEAD;
}

__device__ __forceinline__ const void* weight_map(const FlowArgs& a, int kind, int l) {
  if (kind == K_HEAD) return a.map_head;
  const FlowLayer& w = a.layers[l];
  switch (kind) {
    case K_QKV: return w.map_qkv;
    case K_O: return w.map_o;
    case K_QC: return w.map_qc;
    case K_OC: return w.map_oc;
    case K_FC1: return w.map_fc1;
    default: return w.map_fc2;
  }
}

// FC2 units are ordered slice-major: unit u is row tile u mod (d/16) of slice u / (d/16).
__device__ __forceinline__ int unit_kq(const FlowArgs& a, int kind, int u) { return kind == K_FC2 ? u / (a.d / 16) : 0; }
__device__ __forceinline__ int unit_tile(const FlowArgs& a, int kind, int u) {
  return kind == K_FC2 ? u % (a.d / 16) : u;
}

// Split a CTA's units [s0, s1) of a projection step into bundles: runs of at
// most MAXB tiles of one reduction slice.
template <class F>
__device__ __forceinline__ void bundles(const FlowArgs& a, int kind, int s0, int s1, F&& f) {
  for (int u = s0; u < s1;) {
    const int kq = unit_kq(a, kind, u);
    int e = u + 1;
    while (e < s1 && e - u < MAXB && unit_kq(a, kind, e) == kq) ++e;
    f(u, e);
    u = e;
  }
}

__device__ __forceinline__ int cross_chunks(const Plan& P, int gi) { return max(0, min(4, P.nch_x - 4 * gi)); }

// ------------------------------------------------------------------ producer (warp 0, one lane)
__device__ __noinline__ void producer(const FlowArgs& a, const Plan& P, uint8_t* ring, Smem& sh) {
  uint32_t it = 0;
  bool dead = false;
  auto take = [&](uint32_t bytes) -> int {   // next slot, armed for `bytes`; -1 when aborted
    const int s = (int)(it % NSLOT);
    const uint32_t ph = (it / NSLOT) & 1u;
    if (dead || !ring_wait(a, sh, &sh.empty[s], ph ^ 1u)) { dead = true; return -1; }
    mbar_expect_tx(&sh.full[s], bytes);
    ++it;
    return s;
  };
  walk(a, P, [&](int kind, int l, int s0, int s1) {
    if (dead) return;
    if (is_weight(kind)) {
      const CUtensorMap* map = reinterpret_cast<const CUtensorMap*>(weight_map(a, kind, l));
      for (int u = s0; u < s1; ++u) {
        const int tile = unit_tile(a, kind, u), kq = unit_kq(a, kind, u);
        for (int j = 0; j < P.spt; ++j) {
          const int s = take(SLOT);
          if (s < 0) return;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            tma_load_2d(ring + s * SLOT + i * KB, map, &sh.full[s], kq * a.d + (4 * j + i) * 64, tile * 16);
        }
      }
    } else if (kind == K_SELF) {
      const int h = s0;
      const CUtensorMap* map = reinterpret_cast<const CUtensorMap*>(a.map_kv);
      const size_t layer_rows = a.kv_layer_bytes / (WS_DH * 2);
      const int c_dep = P.L / WS_PAGE;        // chunks from here hold this call's block keys
      for (int c = 0; c < P.nch_self; ++c) {
        if (c == c_dep) {
          if (!wait_ge(a, sh, lctr(a, l, FC_QKV_HEAD + h), 12)) { dead = true; return; }
          fence_async_global();                 // the block's K/V rows were written by other SMs
        }
        const int page = a.ptab[P.slot * a.ppr + c];
        const size_t base = (size_t)l * layer_rows + ((size_t)page * 2 * a.heads + h) * WS_PAGE;
        int s = take(KVBOX);
        if (s < 0) return;
        tma_load_2d(ring + s * SLOT, map, &sh.full[s], 0, (int)base);
        s = take(KVBOX);
        if (s < 0) return;
        tma_load_2d(ring + s * SLOT, map, &sh.full[s], 0, (int)(base + (size_t)a.heads * WS_PAGE));
      }
    } else if (kind == K_CROSS) {
      const int h = s0 / P.ngrp, gi = s0 - h * P.ngrp;
      const CUtensorMap* map = reinterpret_cast<const CUtensorMap*>(a.map_xkv);
      const size_t base = (size_t)P.slot * a.xkv_slot_rows + (size_t)l * a.xkv_layer_rows;
      for (int k = 0; k < cross_chunks(P, gi); ++k) {
        const int fr = (4 * gi + k) * WS_XCHUNK;
        int s = take(KVBOX);
        if (s < 0) return;
        tma_load_2d(ring + s * SLOT, map, &sh.full[s], 0, (int)(base + (size_t)h * a.max_frames + fr));
        s = take(KVBOX);
        if (s < 0) return;
        tma_load_2d(ring + s * SLOT, map, &sh.full[s], 0,
                    (int)(base + (size_t)(a.heads + h) * a.max_frames + fr));
      }
    }
  });
  sh.issued = it;
}

// ------------------------------------------------------------------ compute warps
struct Cursor {
  uint32_t it;      // ring slots consumed
  int btag;         // which B operand bsm holds (-1: none)
  int dtag;         // the last dependency this CTA saw satisfied
  uint32_t bphase;  // parity of the next B-operand copy
  uint32_t xphase;  // parity of the next residual copy
};

__device__ __forceinline__ bool wait_copy(const FlowArgs& a, Smem& sh, uint64_t* bar, int& pending, uint32_t& phase) {
  bool ok = true;
  if (pending) ok = ring_wait(a, sh, bar, phase);
  phase ^= 1u;
  return ok;
}

// B = LayerNorm(x) of the block rows, bf16, laid out [k-block][16 rows][64]
// with the 128-byte swizzle (16-byte chunk c of row t at chunk c ^ (t & 7));
// rows >= H are zero.  The residual rows come in by TMA, xs_rows at a time,
// and are normalised by one warp per row with the layer-norm kernel's
// per-row arithmetic (two-pass fp32 statistics).
__device__ __noinline__ void build_ln(const FlowArgs& a, const Plan& P, const bf16* g, const bf16* b, uint8_t* bsm,
                                      uint8_t* xs, Smem& sh, Cursor& cx) {
  // g, b: gain and bias already staged in shared memory
  const int cw = (threadIdx.x >> 5) - 1, ct = threadIdx.x - 32, lane = threadIdx.x & 31;
  const float* xsf = reinterpret_cast<const float*>(xs);
  for (int p0 = 0; p0 < a.H; p0 += a.xs_rows) {
    if (threadIdx.x == 32 && !sh.abort) {
      fence_async_global();           // residual rows written by other SMs, read by the TMA unit
      fence_async_smem();             // earlier reads of xs come before the copy
      mbar_expect_tx(&sh.xbar, (uint32_t)(a.xs_rows * a.d * 4));
      tma_load_3d(xs, reinterpret_cast<const CUtensorMap*>(a.map_x), &sh.xbar, 0, 0, p0);
      sh.x_pending = 1;
      sh.x_parity = cx.xphase;
    }
    compute_sync();
    const bool ok = wait_copy(a, sh, &sh.xbar, sh.x_pending, cx.xphase);
    const int nrow = min(a.xs_rows, a.H - p0);
    // staged row r on warp r mod 4; per row: per-lane sums over the lane's
    // float4 groups (4 * lane + 128 i) in order, a shuffle tree, then the
    // same for the squared deviations (two-pass statistics), then normalise
    const int nv = a.d >> 7;
#pragma unroll 1
    for (int r = cw; r < nrow && ok; r += 4) {
      const float4* xrow = reinterpret_cast<const float4*>(xsf + (size_t)r * a.d) + lane;
      float sum = 0.f;
#pragma unroll 1
      for (int i = 0; i < nv; ++i) {
        const float4 v = xrow[32 * i];
        sum += (v.x + v.y) + (v.z + v.w);
      }
      const float mean = warp_sum(sum) / (float)a.d;
      float q = 0.f;
#pragma unroll 1
      for (int i = 0; i < nv; ++i) {
        const float4 v = xrow[32 * i];
        const float e0 = v.x - mean, e1 = v.y - mean, e2 = v.z - mean, e3 = v.w - mean;
        q += (e0 * e0 + e1 * e1) + (e2 * e2 + e3 * e3);
      }
      const float rstd = rsqrtf(warp_sum(q) / (float)a.d + 1e-5f);
      const int t = p0 + r;
#pragma unroll 1
      for (int i = 0; i < nv; ++i) {
        const float4 v = xrow[32 * i];
        const int k = 4 * lane + 128 * i, col = k & 63;
        const uint2 gq = *reinterpret_cast<const uint2*>(g + k), bq = *reinterpret_cast<const uint2*>(b + k);
        const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gq.x));
        const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gq.y));
        const float2 b01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bq.x));
        const float2 b23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bq.y));
        __nv_bfloat162 h0 = __floats2bfloat162_rn((v.x - mean) * rstd * g01.x + b01.x, (v.y - mean) * rstd * g01.y + b01.y);
        __nv_bfloat162 h1 = __floats2bfloat162_rn((v.z - mean) * rstd * g23.x + b23.x, (v.w - mean) * rstd * g23.y + b23.y);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t*>(&h0);
        w.y = *reinterpret_cast<uint32_t*>(&h1);
        *reinterpret_cast<uint2*>(bsm + (k >> 6) * KB + t * 128 + ((((col >> 3) ^ (t & 7)) << 4) | ((col & 7) * 2))) =
            w;
      }
    }
    compute_sync();                   // xs free for the next pass; x_pending settled
    if (threadIdx.x == 32 && ok) sh.x_pending = 0;
  }
  const int zr = FLOW_MAX_ROWS - a.H;
  for (int idx = ct; idx < zr * P.kbt * 8; idx += NCT) {
    const int t = a.H + idx / (P.kbt * 8), rem = idx % (P.kbt * 8);
    *reinterpret_cast<uint4*>(bsm + (rem >> 3) * KB + t * 128 + ((rem & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ float bfv(const bf16* p, int i) { return __bfloat162float(p[i]); }

// Epilogue of one projection tile on one warp: lane (g = lane / 4, c = lane %
// 4) holds features g, g + 8 and tokens 2c, 2c + 1, 8 + 2c, 9 + 2c (v[i]:
// feature g + 8 * ((i >> 1) & 1), token 8 * (i >> 2) + 2c + (i & 1)).  Ends
// with the tile's signal (a release add by lane 0 after the warp's stores).
__device__ __noinline__ void epi_head(const FlowArgs& a, Smem& sh, int tile, const float* v) {
  const int lane = threadIdx.x & 31, g = lane >> 2, cq = lane & 3;
#pragma unroll 1
  for (int s = 0; s < 4; ++s) {                 // token 8 (s >> 1) + 2c + (s & 1), features g and g + 8
    const int t = 8 * (s >> 1) + 2 * cq + (s & 1);
    if (t >= a.H) continue;
    unsigned long long key = 0ull;
#pragma unroll 1
    for (int h2 = 0; h2 < 2; ++h2) {
      const int n = tile * 16 + g + 8 * h2;
      if (n >= a.V) continue;
      const bool sup = a.suppress && ((a.suppress[n >> 5] >> (n & 31)) & 1u);
      const float z = sup ? -INFINITY : v[((s >> 1) << 2) | (h2 << 1) | (s & 1)];
      if (a.logits) a.logits[(size_t)t * a.V + n] = z;
      const unsigned long long k = argmax_key(z, n);
      key = k > key ? k : key;
    }
    if (key) atomicMax(&sh.skey[t], key);
  }
}

__device__ __noinline__ void epi_fc2(const FlowArgs& a, const Plan& P, int l, int tile, int kq, const float* v,
                                     const float* bias) {
  const int lane = threadIdx.x & 31, g = lane >> 2, cq = lane & 3;
  const FlowLayer* w = &a.layers[l];
  const int d = a.d;
  {
    float* part = a.fpart + ((size_t)tile * P.ksplit + kq) * 256;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = g + ((i & 2) ? 8 : 0), t = 8 * (i >> 2) + 2 * cq + (i & 1);
      part[f * 16 + t] = v[i];
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atom_acq_rel(lctr(a, l, FC_FC2_ARRIVE + tile), 1) == P.ksplit - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    // every slice of this tile is stored: add them in slice order into the residual
    const float* p0 = a.fpart + (size_t)tile * P.ksplit * 256;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      const int f = g + ((i & 2) ? 8 : 0), t = 8 * (i >> 2) + 2 * cq + (i & 1), n = tile * 16 + f;
      if (t >= a.H) continue;
      float s = __ldcg(p0 + f * 16 + t);
      for (int q = 1; q < P.ksplit; ++q) s += __ldcg(p0 + q * 256 + f * 16 + t);
      float* xp = a.x + (size_t)t * d + n;
      const float y = __ldcg(xp) + (s + bias[(i >> 1) & 1]);
      *xp = y;
      if (w->hist_idx >= 0)
        a.hist[(((size_t)P.slot * a.max_block + t) * a.n_hist + w->hist_idx) * d + n] = y;
    }
    __syncwarp();
    if (lane == 0) red_release(lctr(a, l, FC_FC2_DONE), 1);
  }
}

__device__ __noinline__ void epi_main(const FlowArgs& a, const Plan& P, int kind, int l, int tile, const float* v,
                                      const float* bias, const int* koff) {
  const int lane = threadIdx.x & 31, g = lane >> 2, cq = lane & 3;
  const int d = a.d;
  // residual rows first (all loads of the tile in one round trip), then the stores
  float xr[8];
  if (kind == K_O || kind == K_OC) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = g + ((i & 2) ? 8 : 0), t = 8 * (i >> 2) + 2 * cq + (i & 1), n = tile * 16 + f;
      xr[i] = t < a.H ? __ldcg(a.x + (size_t)t * d + n) : 0.f;
    }
  }
#pragma unroll 1
  for (int i = 0; i < 8; ++i) {
    const int f = g + ((i & 2) ? 8 : 0), t = 8 * (i >> 2) + 2 * cq + (i & 1), n = tile * 16 + f;
    if (t >= a.H) continue;
    const float y = v[i] + bias[(i >> 1) & 1];
    switch (kind) {
      case K_QKV: {
        const int part = n / d, nn = n - part * d;
        if (part == 0) {
          a.q[(size_t)t * d + nn] = __float2bfloat16_rn(y);
        } else {
          const int off = koff[((i >> 2) << 1) | (i & 1)];
          if (off >= 0)
            reinterpret_cast<bf16*>(a.kv + (size_t)l * a.kv_layer_bytes)[off + ((size_t)(part - 1) * a.heads +
                                                                               nn / WS_DH) * (WS_PAGE * WS_DH) +
                                                                        (nn % WS_DH)] = __float2bfloat16_rn(y);
        }
        break;
      }
      case K_QC:
        a.q[(size_t)t * d + n] = __float2bfloat16_rn(y);
        break;
      case K_O:
      case K_OC:
        a.x[(size_t)t * d + n] = xr[i] + y;
        break;
      case K_FC1:
        a.ffn[(size_t)t * a.f + n] = __float2bfloat16_rn(gelu_erf(y));
        break;
      default:
        break;
    }
  }
  __syncwarp();
  if (lane == 0) {
    int* c = nullptr;
    switch (kind) {
      case K_QKV: c = lctr(a, l, FC_QKV_HEAD + ((tile * 16) % d) / WS_DH); break;
      case K_QC: c = lctr(a, l, FC_QC_HEAD + (tile * 16) / WS_DH); break;
      case K_O: c = lctr(a, l, FC_O_DONE); break;
      case K_OC: c = lctr(a, l, FC_OC_DONE); break;
      case K_FC1: c = lctr(a, l, FC_FC1_PIECE + (tile * 16) / d); break;
      default: break;
    }
    if (c) red_release(c, 1);
  }
}

// Counter and target a projection step waits for.
__device__ __forceinline__ const int* dep_of(const FlowArgs& a, int kind, int l, int kq, int& target) {
  const int dt = a.d / 16;
  target = dt;
  switch (kind) {
    case K_QKV: return l == 0 ? gctr(a, FG_EMBED) : lctr(a, l - 1, FC_FC2_DONE);
    case K_O: target = a.heads; return lctr(a, l, FC_SELF_DONE);
    case K_QC: return lctr(a, l, FC_O_DONE);
    case K_OC: target = a.heads; return lctr(a, l, FC_X_DONE);
    case K_FC1: return lctr(a, l, FC_OC_DONE);
    case K_FC2: return lctr(a, l, FC_FC1_PIECE + kq);
    default: return lctr(a, a.n_layers - 1, FC_FC2_DONE);   // K_HEAD
  }
}

__device__ __noinline__ void weight_bundle(const FlowArgs& a, const Plan& P, uint8_t* ring, uint8_t* bsm, uint8_t* xs,
                                           uint8_t* gbs, Smem& sh, Cursor& cx, int kind, int l, int u0, int u1) {
  const int warp = threadIdx.x >> 5, cw = warp - 1, lane = threadIdx.x & 31;
  const int nt = u1 - u0, kq = unit_kq(a, kind, u0);
  const int tag = ((l * 16 + kind) << 4) + kq;
  // ---- constants first (weights and positions: independent of the dependency)
  const bool need_b = cx.btag != tag;
  if (need_b && ln_input(kind)) {
    const bf16 *g, *b;
    if (kind == K_HEAD) { g = a.lnf_g; b = a.lnf_b; }
    else {
      const FlowLayer& w = a.layers[l];
      g = kind == K_QKV ? w.ln1_g : kind == K_QC ? w.ln2_g : w.ln3_g;
      b = kind == K_QKV ? w.ln1_b : kind == K_QC ? w.ln2_b : w.ln3_b;
    }
    const int ct = threadIdx.x - 32, n8 = a.d / 4;          // 8-byte groups of gain + bias
    for (int i = ct; i < 2 * n8; i += NCT) {
      const bf16* src = i < n8 ? g + 4 * i : b + 4 * (i - n8);
      *reinterpret_cast<uint2*>(gbs + 8 * i) = __ldg(reinterpret_cast<const uint2*>(src));
    }
  }
  float bias[2] = {0.f, 0.f};
  int koff[4] = {-1, -1, -1, -1};
  if (cw < nt && kind != K_HEAD) {
    const FlowLayer& w = a.layers[l];
    const int tile = unit_tile(a, kind, u0 + cw), g8 = lane >> 2, cq = lane & 3;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int n = tile * 16 + g8 + 8 * h2;
      const bf16* bp = nullptr;
      int nn = n;
      switch (kind) {
        case K_QKV: {
          const int part = n / a.d;
          nn = n - part * a.d;
          bp = part == 0 ? w.b_q : part == 2 ? w.b_v : nullptr;
          break;
        }
        case K_O: bp = w.b_o; break;
        case K_QC: bp = w.b_qc; break;
        case K_OC: bp = w.b_oc; break;
        case K_FC1: bp = w.b_fc1; break;
        default: bp = w.b_fc2; break;
      }
      bias[h2] = bp ? bfv(bp, nn) : 0.f;
    }
    if (kind == K_QKV) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int t = 8 * (s >> 1) + 2 * cq + (s & 1), pos = P.L + t;
        if (t < a.H && t < P.blen && pos < a.max_pos)
          koff[s] = (int)((size_t)a.ptab[P.slot * a.ppr + pos / WS_PAGE] * 2 * a.heads * (WS_PAGE * WS_DH) +
                          (size_t)(pos % WS_PAGE) * WS_DH);
      }
    }
  }
  // ---- dependency (once per step and slice in this CTA)
  if (cx.dtag != tag) {
    if (threadIdx.x == 32) {
      int target;
      const int* c = dep_of(a, kind, l, kq, target);
      wait_ge(a, sh, c, target);
    }
    cx.dtag = tag;
  }
  compute_sync();
  // ---- B operand: the block rows over this slice, shared by the CTA's bundles of the step
  if (need_b) {
    if (ln_input(kind)) {
      build_ln(a, P, reinterpret_cast<const bf16*>(gbs), reinterpret_cast<const bf16*>(gbs) + a.d, bsm, xs, sh, cx);
    } else {
      if (threadIdx.x == 32 && !sh.abort) {
        const CUtensorMap* map = reinterpret_cast<const CUtensorMap*>(kind == K_FC2 ? a.map_ffn : a.map_ao);
        fence_async_global();           // rows written by other SMs, read by the TMA unit
        fence_async_smem();             // our earlier reads of bsm come before the copy
        mbar_expect_tx(&sh.bbar, (uint32_t)(P.kbt * KB));
        for (int kb = 0; kb < P.kbt; ++kb) tma_load_2d(bsm + kb * KB, map, &sh.bbar, kq * a.d + kb * 64, 0);
        sh.b_pending = 1;
        sh.b_parity = cx.bphase;
      }
      compute_sync();
      const bool ok = wait_copy(a, sh, &sh.bbar, sh.b_pending, cx.bphase);
      compute_sync();
      if (threadIdx.x == 32 && ok) sh.b_pending = 0;
    }
    cx.btag = tag;
  }
  // ---- MMA: warp cw multiplies k-block 4j + cw of every tile (slot j of the
  // tile holds k-blocks 4j .. 4j + 3), four independent accumulator chains
  float* red = reinterpret_cast<float*>(xs);          // [warp][tile][lane][8]
  const int mtx = lane >> 3;
  const int ra = (lane & 7) + ((mtx & 1) ? 8 : 0), tb = (lane & 7) + ((mtx >> 1) ? 8 : 0);
  for (int t = 0; t < nt; ++t) {
    float acc[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[q][i] = 0.f;
    for (int j = 0; j < P.spt; ++j) {
      const uint32_t it = cx.it + (uint32_t)(t * P.spt + j);
      const int s = (int)(it % NSLOT);
      if (ring_wait(a, sh, &sh.full[s], (it / NSLOT) & 1u)) {
        const uint32_t abase = smem_u32(ring + s * SLOT + cw * KB) + (uint32_t)(ra * 128);
        const uint32_t bbase = smem_u32(bsm + (4 * j + cw) * KB) + (uint32_t)(tb * 128);
        uint32_t af[4][4], bf[4][4];
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          ldsm_x4(abase + (((2 * st + (mtx >> 1)) ^ (ra & 7)) << 4), af[st][0], af[st][1], af[st][2], af[st][3]);
          ldsm_x4(bbase + (((2 * st + (mtx & 1)) ^ (tb & 7)) << 4), bf[st][0], bf[st][1], bf[st][2], bf[st][3]);
        }
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          mma_bf16_16816(acc[st], af[st], bf[st][0], bf[st][1]);
          mma_bf16_16816(acc[st] + 4, af[st], bf[st][2], bf[st][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_n(&sh.empty[s], 1);
    }
    float* r = red + (((size_t)cw * MAXB + t) * 32 + lane) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = ((acc[0][i] + acc[1][i]) + acc[2][i]) + acc[3][i];
  }
  compute_sync();
  // ---- the four warps' partial tiles added in warp order; warp t finishes tile t
  if (cw < nt && !sh.abort) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float* r = red + (((size_t)w * MAXB + cw) * 32 + lane) * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += r[i];
    }
    const int u = u0 + cw;
    if (kind == K_HEAD) epi_head(a, sh, unit_tile(a, kind, u), v);
    else if (kind == K_FC2) epi_fc2(a, P, l, unit_tile(a, kind, u), unit_kq(a, kind, u), v, bias);
    else epi_main(a, P, kind, l, unit_tile(a, kind, u), v, bias, koff);
  }
  cx.it += (uint32_t)(nt * P.spt);
}

// The tensor-core partial of one 64-key chunk for the block rows (one warp),
// written to out + r * 66 for rows r < H; one copy of the code for both
// attention kinds.
__device__ __noinline__ void chunk_partial(const uint8_t* Ks, const uint8_t* Vs, const uint32_t (*qf)[4], int vis_lo,
                                           int vis_hi, int nrows, float* out) {
  attn_chunk_partial<true>(Ks, Vs, qf, prefix_mask(vis_lo), prefix_mask(vis_hi), nrows,
                           [&](int r) { return out + (size_t)r * WS_ATTN_PART; });
}

// Combine per-chunk partials (m, l, 64 weighted values) of one row into one
// partial of the same form: M = max m, L = sum l e^(m - M), a = sum a e^(m - M),
// chunks in order.  Lane l handles dims 2l, 2l + 1; out[0..1] by lane 0.
template <class PartOf>
__device__ __forceinline__ void merge_partials(PartOf part_of, int n, float* out) {
  const int lane = threadIdx.x & 31;
  float M = -INFINITY;
  for (int s = 0; s < n; ++s) M = fmaxf(M, part_of(s)[0]);
  float L = 0.f, n0 = 0.f, n1 = 0.f;
  for (int s = 0; s < n; ++s) {
    const float* p = part_of(s);
    if (p[1] <= 0.f) continue;
    const float c = expf(p[0] - M);
    L = fmaf(p[1], c, L);
    n0 = fmaf(p[2 + 2 * lane], c, n0);
    n1 = fmaf(p[3 + 2 * lane], c, n1);
  }
  if (lane == 0) { out[0] = L > 0.f ? M : -INFINITY; out[1] = L; }
  out[2 + 2 * lane] = n0;
  out[3 + 2 * lane] = n1;
}

// Fold of partials into the head's attention output rows (rows cw, cw + 4,
// ...; lane l writes dims 2l, 2l + 1).  GLOBAL: group partials in L2 at
// base + (s * 16 + r) * FLOW_GP, else chunk partials in shared memory at
// base + (s * 16 + r) * 66.
template <bool GLOBAL>
__device__ __noinline__ void fold_rows(const FlowArgs& a, const float* base, int h, int n_split) {
  // partials (m, l, 64 values) of split s, row r at base + (s * 16 + r) * stride;
  // rows cw, cw + 4, ...; lane l writes dims 2l, 2l + 1.  n_split <= 16.
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  constexpr int stride = GLOBAL ? FLOW_GP : WS_ATTN_PART;
#pragma unroll 1
  for (int r = cw; r < a.H; r += 4) {
    const float* p = base + (size_t)r * stride;
    const size_t ss = (size_t)FLOW_MAX_ROWS * stride;
    const float2 ml = lane < n_split ? (GLOBAL ? __ldcg(reinterpret_cast<const float2*>(p + lane * ss))
                                              : *reinterpret_cast<const float2*>(p + lane * ss))
                                     : make_float2(-INFINITY, 0.f);
    const float M = warp_max(ml.x);
    float den = 0.f, n0 = 0.f, n1 = 0.f;
    // splits in order, the value loads of eight splits issued together
#pragma unroll 1
    for (int u0 = 0; u0 < n_split; u0 += 8) {
      float2 av[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (u0 + u < n_split) {
          const float2* q = reinterpret_cast<const float2*>(p + (u0 + u) * ss + 2 + 2 * lane);
          av[u] = GLOBAL ? __ldcg(q) : *q;
        }
#pragma unroll 1
      for (int u = 0; u < 8 && u0 + u < n_split; ++u) {
        const float l = __shfl_sync(0xffffffffu, ml.y, u0 + u), m = __shfl_sync(0xffffffffu, ml.x, u0 + u);
        if (l <= 0.f) continue;
        const float c = expf(m - M);
        den = fmaf(l, c, den);
        n0 = fmaf(av[u].x, c, n0);
        n1 = fmaf(av[u].y, c, n1);
      }
    }
    *reinterpret_cast<__nv_bfloat162*>(a.ao + (size_t)r * a.d + h * WS_DH + 2 * lane) =
        __floats2bfloat162_rn(den > 0.f ? n0 / den : 0.f, den > 0.f ? n1 / den : 0.f);
  }
}

__device__ __noinline__ void self_task(const FlowArgs& a, const Plan& P, uint8_t* ring, uint8_t* bsm, Smem& sh,
                                       Cursor& cx, int l, int h) {
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31, g = lane >> 2;
  if (threadIdx.x == 32) wait_ge(a, sh, lctr(a, l, FC_QKV_HEAD + h), 12);
  compute_sync();
  float* part = reinterpret_cast<float*>(bsm);        // [chunk][16 rows][66]
  uint32_t qf[4][4];
  attn_q_frags(a.q, a.d, 0, a.H, h * WS_DH, qf);
  for (int c = cw; c < P.nch_self; c += 4) {
    const uint32_t ik = cx.it + 2u * c, iv = ik + 1u;
    const int sk = (int)(ik % NSLOT), sv = (int)(iv % NSLOT);
    const bool ok = ring_wait(a, sh, &sh.full[sk], (ik / NSLOT) & 1u) &&
                    ring_wait(a, sh, &sh.full[sv], (iv / NSLOT) & 1u);
    if (ok) {
      const int k0 = c * WS_XCHUNK;
      const int vis_lo = min(max(P.L + g + 1 - k0, 0), WS_XCHUNK);
      const int vis_hi = min(max(P.L + g + 9 - k0, 0), WS_XCHUNK);
      chunk_partial(ring + sk * SLOT, ring + sv * SLOT, qf, vis_lo, vis_hi, a.H,
                    part + (size_t)c * FLOW_MAX_ROWS * WS_ATTN_PART);
    }
    __syncwarp();
    if (lane == 0) { mbar_arrive_n(&sh.empty[sk], 4); mbar_arrive_n(&sh.empty[sv], 4); }
  }
  compute_sync();
  if (!sh.abort) fold_rows<false>(a, part, h, P.nch_self);
  compute_sync();
  if (threadIdx.x == 32) red_release(lctr(a, l, FC_SELF_DONE), 1);
  cx.it += 2u * P.nch_self;
  cx.btag = -1;                       // bsm held the partials
}

__device__ __noinline__ void cross_task(const FlowArgs& a, const Plan& P, uint8_t* ring, uint8_t* xs, Smem& sh,
                                        Cursor& cx, int l, int u) {
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int h = u / P.ngrp, gi = u - h * P.ngrp, nk = cross_chunks(P, gi);
  if (threadIdx.x == 32) wait_ge(a, sh, lctr(a, l, FC_QC_HEAD + h), 4);
  compute_sync();
  float* part = reinterpret_cast<float*>(xs);         // [chunk of the group][16 rows][66]
  if (cw < nk) {
    uint32_t qf[4][4];
    attn_q_frags(a.q, a.d, 0, a.H, h * WS_DH, qf);
    const int c = 4 * gi + cw;
    const uint32_t ik = cx.it + 2u * cw, iv = ik + 1u;
    const int sk = (int)(ik % NSLOT), sv = (int)(iv % NSLOT);
    const bool ok = ring_wait(a, sh, &sh.full[sk], (ik / NSLOT) & 1u) &&
                    ring_wait(a, sh, &sh.full[sv], (iv / NSLOT) & 1u);
    if (ok) {
      const int vis = min(max(P.Fv - c * WS_XCHUNK, 0), WS_XCHUNK);
      chunk_partial(ring + sk * SLOT, ring + sv * SLOT, qf, vis, vis, a.H,
                    part + (size_t)cw * FLOW_MAX_ROWS * WS_ATTN_PART);
    }
    __syncwarp();
    if (lane == 0) { mbar_arrive_n(&sh.empty[sk], 4); mbar_arrive_n(&sh.empty[sv], 4); }
  }
  compute_sync();
  // this group's chunks merged into one partial per row, stored for the head's fold
  float* gp = a.xpart + ((size_t)h * a.max_groups + gi) * FLOW_MAX_ROWS * FLOW_GP;
  for (int r = cw; r < a.H; r += 4)
    merge_partials([&](int s) { return part + ((size_t)s * FLOW_MAX_ROWS + r) * WS_ATTN_PART; }, nk,
                   gp + (size_t)r * FLOW_GP);
  compute_sync();
  if (threadIdx.x == 32) sh.flag = atom_acq_rel(lctr(a, l, FC_X_ARRIVE + h), 1) == P.ngrp - 1;
  compute_sync();
  if (sh.flag) {
    // the head's last group: fold the groups of every row, in group order
    if (!sh.abort) fold_rows<true>(a, a.xpart + (size_t)h * a.max_groups * FLOW_MAX_ROWS * FLOW_GP, h, P.ngrp);
    compute_sync();
    if (threadIdx.x == 32) red_release(lctr(a, l, FC_X_DONE), 1);
  }
  cx.it += 2u * nk;
}

__device__ __noinline__ void embed_task(const FlowArgs& a, const Plan& P, Smem& sh, int e) {
  const int ct = threadIdx.x - 32;
  for (int idx = ct; idx < a.H * 16; idx += NCT) {
    const int t = idx >> 4, n = e * 16 + (idx & 15);
    int pos = P.L + t, tok = a.block[t];
    const bool in_block = t < P.blen;
    if (!(in_block && pos < a.max_pos)) { tok = 0; pos = min(pos, a.max_pos - 1); }
    if (tok < 0 || tok >= a.V) {
      if (e == 0 && (idx & 15) == 0) atomicOr(a.status, WS_ST_TOKEN);
      tok = 0;
    }
    if (e == 0 && (idx & 15) == 0 && in_block && P.L + t >= a.max_pos) atomicOr(a.status, WS_ST_POS);
    a.x[(size_t)t * a.d + n] = bfv(a.tok_emb, tok * a.d + n) + bfv(a.pos_emb, pos * a.d + n);
  }
  if (e == 0) {
    if (ct == 0) { a.pend_start[P.slot] = P.L; a.pend_n[P.slot] = P.blen; }
    if (ct < a.H) a.amax[ct] = 0ull;
  }
  compute_sync();
  if (threadIdx.x == 32) red_release(gctr(a, FG_EMBED), 1);
}

__global__ void __launch_bounds__(NT, 1) flow_verify_kernel(const __grid_constant__ FlowArgs a) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ Smem sh;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  uint8_t* bsm = ring + NSLOT * SLOT;
  uint8_t* xs = bsm + BSM;
  uint8_t* gbs = xs + XS;

  Plan P;
  P.slot = a.req_ids[0];
  P.L = a.L[P.slot];
  P.blen = a.block_len[0];
  P.Fv = a.Fv[P.slot];
  const int ppr_max = (a.max_pos + WS_PAGE - 1) / WS_PAGE;
  P.nch_self = min((P.L + a.H + WS_XCHUNK - 1) / WS_XCHUNK, ppr_max);
  P.nch_x = (P.Fv + WS_XCHUNK - 1) / WS_XCHUNK;
  P.ngrp = max(1, (P.nch_x + 3) / 4);
  P.spt = a.d / 256;
  P.kbt = a.d / 64;
  P.ksplit = a.f / a.d;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) { mbar_init(&sh.full[i], 1); mbar_init(&sh.empty[i], 4); }
    mbar_init(&sh.bbar, 1);
    mbar_init(&sh.xbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sh.abort = 0;
    sh.b_pending = sh.x_pending = 0;
    sh.issued = 0;
  }
  if (threadIdx.x < FLOW_MAX_ROWS) sh.skey[threadIdx.x] = 0ull;
  __syncthreads();

  if (threadIdx.x < 32) {
    if (threadIdx.x == 0) producer(a, P, ring, sh);
  } else {
    Cursor cx{0u, -1, -1, 0u, 0u};
    walk(a, P, [&](int kind, int l, int s0, int s1) {
      if (is_weight(kind)) {
        bundles(a, kind, s0, s1, [&](int u0, int u1) { weight_bundle(a, P, ring, bsm, xs, gbs, sh, cx, kind, l, u0, u1); });
      } else if (kind == K_SELF) {
        self_task(a, P, ring, bsm, sh, cx, l, s0);
      } else if (kind == K_CROSS) {
        cross_task(a, P, ring, xs, sh, cx, l, s0);
      } else {
        embed_task(a, P, sh, s0);
      }
    });
    // LM head: this CTA's row maxima, then the last CTA writes the argmax ids
    compute_sync();
    if (threadIdx.x - 32 < a.H && sh.skey[threadIdx.x - 32] != 0ull)
      atomicMax(a.amax + (threadIdx.x - 32), sh.skey[threadIdx.x - 32]);
    __threadfence();
    compute_sync();
    if (threadIdx.x == 32) sh.flag = atom_acq_rel(gctr(a, FG_HEAD_ARRIVE), 1) == (int)gridDim.x - 1;
    compute_sync();
    if (sh.flag && threadIdx.x - 32 < a.H) {
      const int t = threadIdx.x - 32;
      a.target[t] = t < P.blen ? argmax_key_id(__ldcg(a.amax + t)) : -1;
    }
  }
  __syncthreads();
  // copies still in flight (only after an abort): wait, bounded, for the
  // latest copy issued into each ring slot and for the operand copies
  if (threadIdx.x == 0) {
    for (uint32_t i = sh.issued > (uint32_t)NSLOT ? sh.issued - NSLOT : 0u; i < sh.issued; ++i) {
      const int s = (int)(i % NSLOT);
      const long long t0 = clock64();
      while (!mbar_try_wait(&sh.full[s], (i / NSLOT) & 1u))
        if (clock64() - t0 > SPIN) break;
    }
    const long long t0 = clock64();
    while (sh.b_pending && !mbar_try_wait(&sh.bbar, sh.b_parity))
      if (clock64() - t0 > SPIN) break;
    while (sh.x_pending && !mbar_try_wait(&sh.xbar, sh.x_parity))
      if (clock64() - t0 > 2 * SPIN) break;
    sh.flag = atom_acq_rel(gctr(a, FG_EXIT), 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (sh.flag) {
    // every other CTA is past its last counter access: reset for the next launch
    const int n = a.n_layers * FLOW_CTR_LAYER + FLOW_CTR_GLOBAL;
    for (int i = threadIdx.x; i < n; i += NT) a.ctr[i] = 0;
  }
}

constexpr size_t kSmem = (size_t)NSLOT * SLOT + BSM + XS + GBS + 1024;

}  // namespace

size_t flow_smem_bytes() { return kSmem; }

int flow_prepare() {
  int dev = 0, sms = 0, coop = 0, per = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return 0;
  if (cudaFuncSetAttribute((const void*)flow_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmem) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, flow_verify_kernel, NT, kSmem) != cudaSuccess || per < 1)
    return 0;
  return sms;
}

cudaError_t launch_flow_verify(const FlowArgs& a, int grid, cudaStream_t s) {
  void* args[] = {const_cast<FlowArgs*>(&a)};
  ws_count_launches(1);
  return cudaLaunchCooperativeKernel((const void*)flow_verify_kernel, dim3(grid), dim3(NT), args, kSmem, s);
}
