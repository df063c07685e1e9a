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
// each step is cut into small tasks, dealt to the SMs in a static order, and
// a task waits only for the counters of the tasks whose outputs it reads:
//   * QKV / cross-query projections signal per attention head, so a head's
//     attention starts when its 12 (or 4) tasks are done;
//   * FC2 task (rows, k-slice s) waits only for FC1 slice s;
//   * the output projections wait for all heads, layer norms for the whole
//     residual row (that is what the arithmetic needs).
// Weight streaming does not wait for any of it: warp 0 of each CTA walks the
// CTA's task list and issues TMA loads of every weight tile (and acoustic K/V
// chunk) into a 16-slot shared-memory ring as soon as a slot is free, so HBM
// reads run ahead across steps and layers.
//
// Tasks.  A projection task is 16 output features x one d-wide slice of the
// reduction (FC2's 4d reduction is split into d-wide slices folded in slice
// order by the last-arriving task of the row tile).  Its four compute warps
// each multiply one quarter of the slice with mma.sync m16n8k16 (bf16 in,
// fp32 accumulate; weights as A, the <= 16 block rows as the N = 16 tile),
// the quarters are added in warp order, and the fused epilogue (bias,
// residual, GELU, K/V cache scatter, logits and argmax keys) stores the
// tile.  At <= 16 rows a projection is a weight-streaming GEMV, so the
// legacy warp-level MMA is the right tool here; the tcgen05 engine runs the
// large-batch GEMMs.  Attention reuses the tensor-core chunk partial and the
// fold of the per-op kernels: self-attention of a head in one CTA (its
// chunks on four warps, folded in shared memory), cross-attention in groups
// of four 64-frame chunks per CTA, folded by the head's last-arriving group.
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
constexpr int SLOT = 10240;           // a compute warp's weight quarter (16 x d/4) or one K / V chunk
constexpr int KB = 2048;              // 16 rows x 64 bf16: one k-block of a weight or B tile
constexpr int BSM = 40960;            // B operand [d/64][16][64] bf16, or self-attention partials
constexpr int KVBOX = WS_XCHUNK * WS_DH * 2;   // one 64 x 64 bf16 chunk of K or V
constexpr long long SPIN = 1ll << 31; // clock cycles (~1 s) before a wait gives up

enum Kind { K_EMBED, K_QKV, K_SELF, K_O, K_QC, K_CROSS, K_OC, K_FC1, K_FC2, K_HEAD };

struct Smem {
  uint64_t full[NSLOT], empty[NSLOT], bbar;
  float red[3][32][8];                 // accumulators of compute warps 1..3
  unsigned long long skey[FLOW_MAX_ROWS];
  uint32_t issued;                     // ring slots the producer armed
  int flag;
  int abort;
  int b_pending;                       // a B-operand copy may still be in flight ...
  uint32_t b_parity;                   // ... completing this phase parity of bbar
};

// Per-call quantities every thread derives the same way at kernel start.
struct Plan {
  int slot, L, blen, Fv;
  int nch_self, nch_x, ngrp;
  int kbs, kbt, ksplit;               // k-blocks per warp quarter / per slice; FC2 slices
};

__device__ __forceinline__ int ld_acq(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// AND of a predicate over the 128 compute threads (a barrier of them).
__device__ __forceinline__ bool compute_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, 128, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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
__device__ bool wait_ge(const FlowArgs& a, Smem& sh, const int* p, int target) {
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
__device__ bool ring_wait(const FlowArgs& a, Smem& sh, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (int n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (aborted(a, sh)) return false;
      if (clock64() - t0 > SPIN) { set_abort(a, sh); return false; }
    }
  }
}

// Release / signal: every writing thread fences its global stores, then one
// thread adds to the counter after a barrier of the writers.
__device__ __forceinline__ void signal_after_sync(int* ctr) {
  if (threadIdx.x == 32) atomicAdd(ctr, 1);
}

// The CTA's share of the tasks: stage by stage in dependency order, task u
// of a stage runs on CTA (u + off) mod G where off counts the tasks of all
// earlier stages (so each stage starts where the last one stopped).
template <class F>
__device__ __forceinline__ void walk(const FlowArgs& a, const Plan& P, F&& f) {
  const int G = gridDim.x, b = blockIdx.x;
  int off = 0;
  auto stage = [&](int kind, int layer, int n) {
    for (int u = (b - off % G + G) % G; u < n; u += G) f(kind, layer, u);
    off += n;
  };
  const int dt = a.d / 16;
  stage(K_EMBED, 0, dt);
  for (int l = 0; l < a.n_layers; ++l) {
    stage(K_QKV, l, 3 * dt);
    stage(K_SELF, l, a.heads);
    stage(K_O, l, dt);
    stage(K_QC, l, dt);
    stage(K_CROSS, l, a.heads * P.ngrp);
    stage(K_OC, l, dt);
    stage(K_FC1, l, a.f / 16);
    stage(K_FC2, l, dt * P.ksplit);
  }
  stage(K_HEAD, a.n_layers, (a.V + 15) / 16);
}

__device__ __forceinline__ bool is_weight(int kind) {
  return kind == K_QKV || kind == K_O || kind == K_QC || kind == K_OC || kind == K_FC1 || kind == K_FC2 ||
         kind == K_HEAD;
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

// Row tile and k-slice of a projection task.
__device__ __forceinline__ void task_tile(const FlowArgs& a, int kind, int u, int& tile, int& kq) {
  tile = u;
  kq = 0;
  if (kind == K_FC2) {
    const int dt = a.d / 16;
    kq = u / dt;
    tile = u - kq * dt;
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
  walk(a, P, [&](int kind, int l, int u) {
    if (dead) return;
    if (is_weight(kind)) {
      const CUtensorMap* map = reinterpret_cast<const CUtensorMap*>(weight_map(a, kind, l));
      int tile, kq;
      task_tile(a, kind, u, tile, kq);
      for (int w = 0; w < 4; ++w) {
        const int s = take((uint32_t)(P.kbs * KB));
        if (s < 0) return;
        for (int kb = 0; kb < P.kbs; ++kb)
          tma_load_2d(ring + s * SLOT + kb * KB, map, &sh.full[s], kq * a.d + (w * P.kbs + kb) * 64, tile * 16);
      }
    } else if (kind == K_SELF) {
      const int h = u;
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
      const int h = u / P.ngrp, gi = u - h * P.ngrp;
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
  uint32_t bphase;  // parity of the next B-operand copy
};

// B = LayerNorm(x) of the block rows, bf16, laid out [k-block][16 rows][64]
// with the 128-byte swizzle (16-byte chunk c of row t at chunk c ^ (t & 7));
// rows >= H are zero.  Rows cw, cw + 4, ... are normalised by compute warp
// cw with the per-row warp arithmetic of the layer-norm kernel.
__device__ __noinline__ void build_ln(const FlowArgs& a, const Plan& P, const bf16* g, const bf16* b, uint8_t* bsm) {
  const int cw = (threadIdx.x >> 5) - 1, ct = threadIdx.x - 32;
  // rows cw, cw + 4, cw + 8 in one memory round trip (block rows <= 12), then cw + 12
  for (int r0 = 0; r0 < a.H; r0 += 12) {
    const int first = r0 + cw;
    const int nr = a.H > first ? min(3, (a.H - first + 3) >> 2) : 0;
    const float* xs[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) xs[j] = a.x + (size_t)(first + 4 * j) * a.d;   // read for j < nr only
    ln_rows_warp<true, 3, 10>(xs, nr, a.d, g, b, true, [&](int j, int k, float v0, float v1, float v2, float v3) {
      const int t = first + 4 * j, col = k & 63;
      __nv_bfloat162 h0 = __floats2bfloat162_rn(v0, v1), h1 = __floats2bfloat162_rn(v2, v3);
      uint2 w;
      w.x = *reinterpret_cast<uint32_t*>(&h0);
      w.y = *reinterpret_cast<uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(bsm + (k >> 6) * KB + t * 128 + ((((col >> 3) ^ (t & 7)) << 4) | ((col & 7) * 2))) =
          w;
    });
  }
  const int zr = FLOW_MAX_ROWS - a.H;
  for (int idx = ct; idx < zr * P.kbt * 8; idx += NCT) {
    const int t = a.H + idx / (P.kbt * 8), rem = idx % (P.kbt * 8);
    *reinterpret_cast<uint4*>(bsm + (rem >> 3) * KB + t * 128 + ((rem & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ float bfv(const bf16* p, int i) { return __bfloat162float(p[i]); }

// Epilogue of one projection task: compute warp 0 holds the summed tile,
// lane (g = lane / 4, c = lane % 4) the values of features g, g + 8 and
// tokens 2c, 2c + 1, 8 + 2c, 9 + 2c (v[i]: feature g + 8 * ((i >> 1) & 1),
// token 8 * (i >> 2) + 2c + (i & 1)).
__device__ __noinline__ void epilogue(const FlowArgs& a, const Plan& P, Smem& sh, int kind, int l, int tile, int kq,
                         const float* v) {
  const int lane = threadIdx.x & 31, g = lane >> 2, cq = lane & 3;
  const FlowLayer* w = kind == K_HEAD ? nullptr : &a.layers[l];
  const int d = a.d;
  if (kind == K_HEAD) {
    unsigned long long key[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = g + ((i & 2) ? 8 : 0), t = 8 * (i >> 2) + 2 * cq + (i & 1), n = tile * 16 + f;
      if (n < a.V && t < a.H) {
        const bool sup = a.suppress && ((a.suppress[n >> 5] >> (n & 31)) & 1u);
        const float z = sup ? -INFINITY : v[i];
        if (a.logits) a.logits[(size_t)t * a.V + n] = z;
        const unsigned long long k = argmax_key(z, n);
        const int s = ((i >> 2) << 1) | (i & 1);
        key[s] = k > key[s] ? k : key[s];
      }
    }
    // reduce over the 8 lanes that hold the same tokens (g = 0..7)
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, key[s], o);
        key[s] = other > key[s] ? other : key[s];
      }
    }
    if (g == 0) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int t = 8 * (s >> 1) + 2 * cq + (s & 1);
        if (key[s] > sh.skey[t]) sh.skey[t] = key[s];
      }
    }
    return;
  }
  if (kind == K_FC2) {
    float* part = a.fpart + ((size_t)tile * P.ksplit + kq) * 256;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = g + ((i & 2) ? 8 : 0), t = 8 * (i >> 2) + 2 * cq + (i & 1);
      part[f * 16 + t] = v[i];
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(lctr(a, l, FC_FC2_ARRIVE + tile), 1) == P.ksplit - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    const float* p0 = a.fpart + (size_t)tile * P.ksplit * 256;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = g + ((i & 2) ? 8 : 0), t = 8 * (i >> 2) + 2 * cq + (i & 1), n = tile * 16 + f;
      if (t >= a.H) continue;
      float s = __ldcg(p0 + f * 16 + t);
      for (int q = 1; q < P.ksplit; ++q) s += __ldcg(p0 + q * 256 + f * 16 + t);
      float* xp = a.x + (size_t)t * d + n;
      const float y = __ldcg(xp) + (s + bfv(w->b_fc2, n));
      *xp = y;
      if (w->hist_idx >= 0)
        a.hist[(((size_t)P.slot * a.max_block + t) * a.n_hist + w->hist_idx) * d + n] = y;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(lctr(a, l, FC_FC2_DONE), 1);
    return;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int f = g + ((i & 2) ? 8 : 0), t = 8 * (i >> 2) + 2 * cq + (i & 1), n = tile * 16 + f;
    if (t >= a.H) continue;
    switch (kind) {
      case K_QKV: {
        const int part = n / d, nn = n - part * d;
        if (part == 0) {
          a.q[(size_t)t * d + nn] = __float2bfloat16_rn(v[i] + bfv(w->b_q, nn));
        } else {
          const int pos = P.L + t;
          if (t < P.blen && pos < a.max_pos) {
            const int page = a.ptab[P.slot * a.ppr + pos / WS_PAGE];
            bf16* kv = reinterpret_cast<bf16*>(a.kv + (size_t)l * a.kv_layer_bytes) +
                       (((size_t)page * 2 + (part - 1)) * a.heads + nn / WS_DH) * (WS_PAGE * WS_DH) +
                       (size_t)(pos % WS_PAGE) * WS_DH + (nn % WS_DH);
            *kv = __float2bfloat16_rn(part == 2 ? v[i] + bfv(w->b_v, nn) : v[i]);
          }
        }
        break;
      }
      case K_QC:
        a.q[(size_t)t * d + n] = __float2bfloat16_rn(v[i] + bfv(w->b_qc, n));
        break;
      case K_O:
      case K_OC: {
        float* xp = a.x + (size_t)t * d + n;
        *xp = __ldcg(xp) + (v[i] + bfv(kind == K_O ? w->b_o : w->b_oc, n));
        break;
      }
      case K_FC1:
        a.ffn[(size_t)t * a.f + n] = __float2bfloat16_rn(gelu_erf(v[i] + bfv(w->b_fc1, n)));
        break;
      default:
        break;
    }
  }
  __threadfence();
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
    if (c) atomicAdd(c, 1);
  }
}

__device__ __noinline__ void weight_task(const FlowArgs& a, const Plan& P, uint8_t* ring, uint8_t* bsm, Smem& sh, Cursor& cx,
                            int kind, int l, int u) {
  const int warp = threadIdx.x >> 5, cw = warp - 1, lane = threadIdx.x & 31;
  int tile, kq;
  task_tile(a, kind, u, tile, kq);
  // ---- dependency
  if (threadIdx.x == 32) {
    const int dt = a.d / 16;
    switch (kind) {
      case K_QKV: wait_ge(a, sh, l == 0 ? gctr(a, FG_EMBED) : lctr(a, l - 1, FC_FC2_DONE), dt); break;
      case K_O: wait_ge(a, sh, lctr(a, l, FC_SELF_DONE), a.heads); break;
      case K_QC: wait_ge(a, sh, lctr(a, l, FC_O_DONE), dt); break;
      case K_OC: wait_ge(a, sh, lctr(a, l, FC_X_DONE), a.heads); break;
      case K_FC1: wait_ge(a, sh, lctr(a, l, FC_OC_DONE), dt); break;
      case K_FC2: wait_ge(a, sh, lctr(a, l, FC_FC1_PIECE + kq), dt); break;
      default: wait_ge(a, sh, lctr(a, a.n_layers - 1, FC_FC2_DONE), dt); break;   // K_HEAD
    }
  }
  compute_sync();
  // ---- B operand (the block rows over this task's k-slice), shared by the
  // CTA's tasks of the same step
  const int tag = ((l * 16 + kind) << 4) + kq;
  if (cx.btag != tag) {
    if (kind == K_QKV || kind == K_QC || kind == K_FC1 || kind == K_HEAD) {
      const bf16 *g, *b;
      if (kind == K_HEAD) { g = a.lnf_g; b = a.lnf_b; }
      else {
        const FlowLayer& w = a.layers[l];
        g = kind == K_QKV ? w.ln1_g : kind == K_QC ? w.ln2_g : w.ln3_g;
        b = kind == K_QKV ? w.ln1_b : kind == K_QC ? w.ln2_b : w.ln3_b;
      }
      build_ln(a, P, g, b, bsm);
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
      const bool issued = sh.b_pending != 0;
      bool landed = true;
      if (issued) landed = ring_wait(a, sh, &sh.bbar, cx.bphase);
      if (issued) cx.bphase ^= 1u;
      landed = compute_and(landed);
      if (threadIdx.x == 32 && landed) sh.b_pending = 0;
    }
    compute_sync();
    cx.btag = tag;
  }
  // ---- MMA: compute warp cw multiplies ring slot it + cw (k-blocks cw * kbs ..)
  const uint32_t it = cx.it + (uint32_t)cw;
  const int s = (int)(it % NSLOT);
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
  if (ring_wait(a, sh, &sh.full[s], (it / NSLOT) & 1u)) {
    const int mtx = lane >> 3;
    const int ra = (lane & 7) + ((mtx & 1) ? 8 : 0), tb = (lane & 7) + ((mtx >> 1) ? 8 : 0);
    const uint32_t abase = smem_u32(ring + s * SLOT) + (uint32_t)(ra * 128);
    const uint32_t bbase = smem_u32(bsm) + (uint32_t)(cw * P.kbs * KB + tb * 128);
#pragma unroll 1
    for (int kb = 0; kb < P.kbs; ++kb) {
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        uint32_t af[4], b0, b1, b2, b3;
        ldsm_x4(abase + kb * KB + ((((2 * st + (mtx >> 1)) ^ (ra & 7))) << 4), af[0], af[1], af[2], af[3]);
        ldsm_x4(bbase + kb * KB + ((((2 * st + (mtx & 1)) ^ (tb & 7))) << 4), b0, b1, b2, b3);
        mma_bf16_16816(c0, af, b0, b1);
        mma_bf16_16816(c1, af, b2, b3);
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive1(&sh.empty[s]);
  // ---- quarters added in warp order, then the epilogue on compute warp 0
  if (cw > 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) { sh.red[cw - 1][lane][i] = c0[i]; sh.red[cw - 1][lane][4 + i] = c1[i]; }
  }
  compute_sync();
  if (cw == 0) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) { v[i] = c0[i]; v[4 + i] = c1[i]; }
#pragma unroll
    for (int r = 0; r < 3; ++r) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += sh.red[r][lane][i];
    }
    if (!sh.abort) epilogue(a, P, sh, kind, l, tile, kq, v);
  }
  cx.it += 4;
}

// Fold of per-chunk partials into the head's attention output rows (rows
// cw, cw + 4, ...; lane l writes dims 2l, 2l + 1).  GLOBAL: partials in L2
// at base + (r * heads + h) * max_xchunks * 66, else in shared memory at
// base + (chunk * 16 + r) * 66.
template <bool GLOBAL>
__device__ __noinline__ void fold_rows(const FlowArgs& a, const float* base, int h, int n_split) {
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  for (int r = cw; r < a.H; r += 4) {
    float o0, o1;
    if (GLOBAL)
      attn_fold_row<true>(base + ((size_t)r * a.heads + h) * a.max_xchunks * WS_ATTN_PART, n_split, o0, o1);
    else
      attn_fold_row_of<false, false>([&](int sp) { return base + ((size_t)sp * FLOW_MAX_ROWS + r) * WS_ATTN_PART; },
                                     n_split, o0, o1);
    *reinterpret_cast<__nv_bfloat162*>(a.ao + (size_t)r * a.d + h * WS_DH + 2 * lane) =
        __floats2bfloat162_rn(o0, o1);
  }
}

__device__ __noinline__ void self_task(const FlowArgs& a, const Plan& P, uint8_t* ring, uint8_t* bsm, Smem& sh, Cursor& cx,
                          int l, int h) {
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
      attn_chunk_partial<true>(ring + sk * SLOT, ring + sv * SLOT, qf, vis_lo, vis_hi, a.H,
                               [&](int r) { return part + ((size_t)c * FLOW_MAX_ROWS + r) * WS_ATTN_PART; });
    }
    __syncwarp();
    if (lane == 0) { mbar_arrive1(&sh.empty[sk]); mbar_arrive1(&sh.empty[sv]); }
  }
  compute_sync();
  if (!sh.abort) fold_rows<false>(a, part, h, P.nch_self);
  __threadfence();
  compute_sync();
  signal_after_sync(lctr(a, l, FC_SELF_DONE));
  cx.it += 2u * P.nch_self;
  cx.btag = -1;                       // bsm held the partials
}

__device__ __noinline__ void cross_task(const FlowArgs& a, const Plan& P, uint8_t* ring, Smem& sh, Cursor& cx, int l, int u) {
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int h = u / P.ngrp, gi = u - h * P.ngrp, nk = cross_chunks(P, gi);
  if (threadIdx.x == 32) wait_ge(a, sh, lctr(a, l, FC_QC_HEAD + h), 4);
  compute_sync();
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
      attn_chunk_partial<true>(ring + sk * SLOT, ring + sv * SLOT, qf, vis, vis, a.H, [&](int r) {
        return a.xpart + (((size_t)r * a.heads + h) * a.max_xchunks + c) * WS_ATTN_PART;
      });
    }
    __syncwarp();
    if (lane == 0) { mbar_arrive1(&sh.empty[sk]); mbar_arrive1(&sh.empty[sv]); }
  }
  __threadfence();
  compute_sync();
  if (threadIdx.x == 32) sh.flag = atomicAdd(lctr(a, l, FC_X_ARRIVE + h), 1) == P.ngrp - 1;
  compute_sync();
  if (sh.flag) {
    // the head's last group: fold every chunk partial of every row, in chunk order
    __threadfence();
    if (!sh.abort) fold_rows<true>(a, a.xpart, h, P.nch_x);
    __threadfence();
    compute_sync();
    signal_after_sync(lctr(a, l, FC_X_DONE));
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
  __threadfence();
  compute_sync();
  signal_after_sync(gctr(a, FG_EMBED));
}

__global__ void __launch_bounds__(NT, 1) flow_verify_kernel(const __grid_constant__ FlowArgs a) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ Smem sh;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  uint8_t* bsm = ring + NSLOT * SLOT;

  Plan P;
  P.slot = a.req_ids[0];
  P.L = a.L[P.slot];
  P.blen = a.block_len[0];
  P.Fv = a.Fv[P.slot];
  const int ppr_max = (a.max_pos + WS_PAGE - 1) / WS_PAGE;
  P.nch_self = min((P.L + a.H + WS_XCHUNK - 1) / WS_XCHUNK, ppr_max);
  P.nch_x = (P.Fv + WS_XCHUNK - 1) / WS_XCHUNK;
  P.ngrp = max(1, (P.nch_x + 3) / 4);
  P.kbs = a.d / 256;
  P.kbt = a.d / 64;
  P.ksplit = a.f / a.d;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) { mbar_init(&sh.full[i], 1); mbar_init(&sh.empty[i], 1); }
    mbar_init(&sh.bbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sh.abort = 0;
    sh.b_pending = 0;
    sh.issued = 0;
  }
  if (threadIdx.x < FLOW_MAX_ROWS) sh.skey[threadIdx.x] = 0ull;
  __syncthreads();

  if (threadIdx.x < 32) {
    if (threadIdx.x == 0) producer(a, P, ring, sh);
  } else {
    Cursor cx{0u, -1, 0u};
    walk(a, P, [&](int kind, int l, int u) {
      if (is_weight(kind)) weight_task(a, P, ring, bsm, sh, cx, kind, l, u);
      else if (kind == K_SELF) self_task(a, P, ring, bsm, sh, cx, l, u);
      else if (kind == K_CROSS) cross_task(a, P, ring, sh, cx, l, u);
      else embed_task(a, P, sh, u);
    });
    // LM head: this CTA's row maxima, then the last CTA writes the argmax ids
    compute_sync();
    if (threadIdx.x - 32 < a.H && sh.skey[threadIdx.x - 32] != 0ull)
      atomicMax(a.amax + (threadIdx.x - 32), sh.skey[threadIdx.x - 32]);
    __threadfence();
    compute_sync();
    if (threadIdx.x == 32) {
      sh.flag = atomicAdd(gctr(a, FG_HEAD_ARRIVE), 1) == (int)gridDim.x - 1;
    }
    compute_sync();
    if (sh.flag && threadIdx.x - 32 < a.H) {
      __threadfence();
      const int t = threadIdx.x - 32;
      a.target[t] = t < P.blen ? argmax_key_id(__ldcg(a.amax + t)) : -1;
    }
  }
  __syncthreads();
  // copies still in flight (only after an abort): wait, bounded, for the
  // latest copy issued into each ring slot
  if (threadIdx.x == 0) {
    for (uint32_t i = sh.issued > (uint32_t)NSLOT ? sh.issued - NSLOT : 0u; i < sh.issued; ++i) {
      const int s = (int)(i % NSLOT);
      const long long t0 = clock64();
      while (!mbar_try_wait(&sh.full[s], (i / NSLOT) & 1u))
        if (clock64() - t0 > SPIN) break;
    }
    if (sh.b_pending) {
      const long long t0 = clock64();
      while (!mbar_try_wait(&sh.bbar, sh.b_parity))
        if (clock64() - t0 > SPIN) break;
    }
    __threadfence();
    sh.flag = atomicAdd(gctr(a, FG_EXIT), 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (sh.flag) {
    // every other CTA is past its last counter access: reset for the next launch
    __threadfence();
    const int n = a.n_layers * FLOW_CTR_LAYER + FLOW_CTR_GLOBAL;
    for (int i = threadIdx.x; i < n; i += NT) a.ctr[i] = 0;
  }
}

constexpr size_t kSmem = (size_t)NSLOT * SLOT + BSM + 1024;

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
