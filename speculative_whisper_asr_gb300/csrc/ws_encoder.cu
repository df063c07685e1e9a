// Whisper audio encoder on the GPU (bf16): the step before the decoding
// path.  Once speculation removes most decoder calls the fixed encoder cost
// shows (Whisper-Flash App. B.2, Table A2: 15-34% of request time at batch
// one, about half at batch 32-96), so it runs here as well.
//
// The pages name the encoder but do not print its layers; this is the
// published Whisper audio encoder:
//   conv1 (n_mels -> d, kernel 3, pad 1) + GELU, conv2 (d -> d, kernel 3,
//   stride 2, pad 1) + GELU, + sinusoidal positions, n_layers pre-LN blocks
//   (non-causal attention over all frames, GELU MLP), final layer norm.
//
// Every projection, both convolutions included, is a tcgen05 GEMM of the
// decoder's engine (ws_gemm_tc.cu) with a fused bias / GELU / residual
// epilogue.  The convolutions become GEMMs over an im2col matrix (conv1:
// [2F, 3 n_mels] padded to a multiple of 64 columns; conv2: [F, 3d], whose
// row t is rows 2t-1 .. 2t+1 of conv1's output).  Attention is a
// flash-attention kernel: one CTA per (64 query rows, head, window), K/V
// tiles of 64 keys double-buffered by TMA, S = Q K^T and O += P V on
// mma.sync with an fp32 online softmax.  Several windows run as one batch
// of n * F rows.
#include <cuda.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "ws_attn_mma.cuh"
#include "ws_internal.cuh"
#include "ws_tc.cuh"

struct EncLayer {
  const bf16 *w_qkv, *w_o, *w_fc1, *w_fc2;
  TcMap m_qkv, m_o, m_fc1, m_fc2;
  const bf16 *b_o, *b_fc1, *b_fc2;
  bf16* b_qkv;                  // [3d]: b_q | 0 | b_v
  const bf16 *ln1_g, *ln1_b, *ln2_g, *ln2_b;
};

struct ws_enc {
  ws_encoder_desc d;
  int kp = 0;                   // im2col width of conv1 (3 n_mels rounded up to 64)
  bf16 *w1 = nullptr, *w2 = nullptr;          // repacked convolution weights [d, kp], [d, 3d]
  TcMap m_w1, m_w2;
  const bf16 *b1 = nullptr, *b2 = nullptr, *lnp_g = nullptr, *lnp_b = nullptr;
  std::vector<EncLayer> layers;
  float* pos = nullptr;         // [F, d] position table
  bf16 *x1 = nullptr, *h1 = nullptr, *x2 = nullptr, *h = nullptr, *qkv = nullptr, *ao = nullptr, *ffn = nullptr;
  float* x = nullptr;           // residual stream [B F, d]
  int32_t* status = nullptr;
  std::map<std::tuple<const void*, int, int>, TcMap> maps;   // activation maps by (base, rows, token tile)
  int attn_tc = 1;              // attention on tcgen05 (1) or on mma.sync (0)
  std::string err;
};

namespace {

thread_local std::string g_enc_err;

int efail(ws_enc* e, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (e) e->err = buf; else g_enc_err = buf;
  return code;
}

#define ECK(x)                                                                                   \
  do {                                                                                           \
    cudaError_t e_ = (x);                                                                        \
    if (e_ != cudaSuccess) return efail(e, WS_ECUDA, "%s: %s", #x, cudaGetErrorString(e_));      \
  } while (0)

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

const char* check_enc_desc(const ws_encoder_desc* d) {
  if (!d) return "null encoder description";
  if (d->n_layers < 1 || d->n_layers > 128) return "n_layers out of range";
  if (d->d_model < 128 || d->d_model % 128 != 0 || d->d_model > 2048) return "d_model must be a multiple of 128, <= 2048";
  if (d->n_heads < 1 || d->d_model % d->n_heads != 0 || d->d_model / d->n_heads != WS_DH) return "d_model / n_heads must be 64";
  if (d->d_ff < 128 || d->d_ff % 128 != 0) return "d_ff must be a multiple of 128";
  if (d->n_mels < 1 || d->n_mels > 1024) return "n_mels out of range";
  if (d->n_frames < 1 || d->n_frames > 16384) return "n_frames out of range";
  if (d->max_batch < 1 || d->max_batch > 256) return "max_batch out of range";
  return nullptr;
}

// Blob element count (see ws.h).
size_t blob_elems(const ws_encoder_desc& d) {
  const size_t D = d.d_model, F = d.d_ff;
  const size_t layer = 3 * D * D + 2 * D + D * D + D + 4 * D + F * D + F + D * F + D;
  return D * d.n_mels * 3 + D + D * D * 3 + D + (size_t)d.n_layers * layer + 2 * D;
}

struct EncPlan {
  size_t blob, w1, w2, bqkv, pos, x1, h1, x2, x, h, qkv, ao, ffn, status, total;
};

EncPlan plan(const ws_encoder_desc& d) {
  EncPlan p;
  const size_t D = d.d_model, B = d.max_batch, F = d.n_frames, T = 2 * F;
  const size_t kp = (3 * (size_t)d.n_mels + 63) / 64 * 64;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = up256(off + bytes); return o; };
  p.blob = take(blob_elems(d) * 2);
  p.w1 = take(D * kp * 2);
  p.w2 = take(D * 3 * D * 2);
  p.bqkv = take((size_t)d.n_layers * 3 * D * 2);
  p.pos = take(F * D * 4);
  p.x1 = take(B * T * kp * 2);
  p.h1 = take(B * T * D * 2);
  p.x2 = take(B * F * 3 * D * 2);
  p.x = take(B * F * D * 4);
  p.h = take(B * F * D * 2);
  p.qkv = take(B * F * 3 * D * 2);
  p.ao = take(B * F * D * 2);
  p.ffn = take(B * F * (size_t)d.d_ff * 2);
  p.status = take(256);
  p.total = off;
  return p;
}

cudaLaunchConfig_t cfg_of(dim3 grid, dim3 block, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.dynamicSmemBytes = smem;
  c.stream = s;
  return c;
}

// ------------------------------------------------------------------ set-up kernels
// dst[o, k * c_in + c] = src[o, c, k] (torch Conv1d layout -> im2col order);
// columns >= 3 c_in are zero.
__global__ void conv_repack_kernel(const bf16* src, bf16* dst, int c_out, int c_in, int kp) {
  const size_t total = (size_t)c_out * kp;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const int o = (int)(idx / kp), col = (int)(idx % kp);
    bf16 v = __float2bfloat16_rn(0.0f);
    if (col < 3 * c_in) {
      const int k = col / c_in, c = col - k * c_in;
      v = src[((size_t)o * c_in + c) * 3 + k];
    }
    dst[idx] = v;
  }
}

// b_qkv of one layer: b_q | 0 | b_v (no key bias).
__global__ void qkv_bias_kernel(const bf16* bq, const bf16* bv, bf16* out, int d) {
  for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < 3 * d; n += gridDim.x * blockDim.x) {
    bf16 v = __float2bfloat16_rn(0.0f);
    if (n < d) v = bq[n];
    else if (n >= 2 * d) v = bv[n - 2 * d];
    out[n] = v;
  }
}

// P[t, i] = sin(t w_i), P[t, d/2 + i] = cos(t w_i), w_i = 10000^(-i / (d/2 - 1)),
// evaluated in double and rounded once.
__global__ void enc_pos_table_kernel(float* pos, int F, int d) {
  const int half = d / 2;
  const size_t total = (size_t)F * half;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(idx / half), i = (int)(idx % half);
    const double w = exp(-(double)i * (log(10000.0) / (double)(half - 1)));
    const double a = (double)t * w;
    pos[(size_t)t * d + i] = (float)sin(a);
    pos[(size_t)t * d + half + i] = (float)cos(a);
  }
}

// ------------------------------------------------------------------ stem kernels
// im2col of conv1: X1[i T + t, k n_mels + c] = mel[i, c, t + k - 1] (zero
// outside 0..T-1 and in the padding columns).  One CTA per row.
__global__ void im2col1_kernel(const bf16* mel, bf16* x1, int n_mels, int T, int kp) {
  const int r = blockIdx.x, i = r / T, t = r - i * T;
  const bf16* m = mel + (size_t)i * n_mels * T;
  for (int col = threadIdx.x; col < kp; col += blockDim.x) {
    bf16 v = __float2bfloat16_rn(0.0f);
    if (col < 3 * n_mels) {
      const int k = col / n_mels, c = col - k * n_mels, src = t + k - 1;
      if (src >= 0 && src < T) v = m[(size_t)c * T + src];
    }
    x1[(size_t)r * kp + col] = v;
  }
}

// im2col of conv2: X2[i F + t, k d + c] = H1[i T + 2t + k - 1, c] (zero
// outside 0..T-1).  16-byte copies; one CTA per row.
__global__ void im2col2_kernel(const bf16* h1, bf16* x2, int d, int F) {
  const int r = blockIdx.x, i = r / F, t = r - i * F, T = 2 * F;
  const int vec = d / 8;                          // 16-byte chunks per source row
  for (int idx = threadIdx.x; idx < 3 * vec; idx += blockDim.x) {
    const int k = idx / vec, c8 = idx - k * vec, src = 2 * t + k - 1;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (src >= 0 && src < T) v = reinterpret_cast<const uint4*>(h1 + ((size_t)i * T + src) * d)[c8];
    reinterpret_cast<uint4*>(x2 + (size_t)r * 3 * d)[idx] = v;
  }
}

// Residual stream x[i F + t, c] = H2[i F + t, c] + P[t, c] (fp32).
__global__ void add_pos_kernel(const bf16* h2, const float* pos, float* x, int d, int F, size_t total) {
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const size_t r = idx / d;
    const int c = (int)(idx - r * d), t = (int)(r % F);
    x[idx] = __bfloat162float(h2[idx]) + pos[(size_t)t * d + c];
  }
}

// ------------------------------------------------------------------ attention
// Non-causal multi-head attention of each window: out[i F + q, h 64 + :] =
// softmax_k(Q_q . K_k / 8) V_k over the window's F keys.  CTA (64 query
// rows, head, window), 4 warps of 16 rows.  K and V tiles of 64 keys arrive
// by TMA (64 x 64 boxes of the [rows, 3d] QKV matrix, 128-byte swizzle) into
// two stages; keys past the window (the next window's rows, or past the
// matrix: zeros) are masked.  Row state: running max m, sum l and the fp32
// accumulator; P enters the second product as bf16.
constexpr int EA_STAGE = 2 * WS_XCHUNK * WS_DH * 2;        // K + V of one tile, 16 KB
constexpr int EA_SMEM = 2 * EA_STAGE + 1024;
constexpr long long EA_WAIT = 1ll << 32;

__device__ __forceinline__ bool ea_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_addr_u32(bar)), "r"(parity) : "memory");
    if (ok) return true;
    if (clock64() - t0 > EA_WAIT) return false;
  }
}

__device__ __forceinline__ void ea_load_tile(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int xk, int xv,
                                             int y) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr_u32(bar)), "r"(EA_STAGE)
               : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr_u32(dst)), "l"((uint64_t)map), "r"(xk), "r"(y), "r"(smem_addr_u32(bar)) : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr_u32(dst + EA_STAGE / 2)), "l"((uint64_t)map), "r"(xv), "r"(y), "r"(smem_addr_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(128) enc_attn_kernel(const __grid_constant__ CUtensorMap tmQKV, const bf16* qkv,
                                                       bf16* out, int F, int d, int32_t* status) {
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t bar[2];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int tile = blockIdx.x, h = blockIdx.y, i = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int row0 = i * F, q0 = tile * 64 + warp * 16;
  const int nrows = max(0, min(16, F - q0));
  const int n_tiles = (F + WS_XCHUNK - 1) / WS_XCHUNK;
  const int xk = d + h * WS_DH, xv = 2 * d + h * WS_DH;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr_u32(&bar[0])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr_u32(&bar[1])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) ea_load_tile(&tmQKV, base, &bar[0], xk, xv, row0);
  uint32_t qf[4][4];
  attn_q_frags(qkv, 3 * d, row0 + q0, nrows, h * WS_DH, qf);
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  int failed = -1;                      // tile whose copy did not land in time
  for (int kt = 0; kt < n_tiles; ++kt) {
    const int st = kt & 1;
    if (threadIdx.x == 0 && kt + 1 < n_tiles)
      ea_load_tile(&tmQKV, base + (st ^ 1) * EA_STAGE, &bar[st ^ 1], xk, xv, row0 + (kt + 1) * WS_XCHUNK);
    const bool landed = ea_wait(&bar[st], (uint32_t)((kt >> 1) & 1));
    if (!__syncthreads_and(landed)) { failed = kt; break; }    // the whole CTA leaves together
    const uint32_t kb = smem_addr_u32(base + st * EA_STAGE), vb = kb + EA_STAGE / 2;
    const int nvis = min(WS_XCHUNK, F - kt * WS_XCHUNK);   // keys of this tile inside the window
    // ---- S = Q K^T / 8
    float sc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 4; s2 += 2) {
        const int mtx = lane >> 3, rr = lane & 7;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + kv_off<true>(8 * j + rr, 2 * s2 + mtx), b0, b1, b2, b3);
        mma_bf16_16816(sc[j], qf[s2], b0, b1);
        mma_bf16_16816(sc[j], qf[s2 + 1], b2, b3);
      }
    }
    // ---- online softmax (rows g and g + 8 of the warp)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = 8 * j + 2 * c + e;
        sc[j][e] = key < nvis ? sc[j][e] * 0.125f : -INFINITY;
        sc[j][2 + e] = key < nvis ? sc[j][2 + e] * 0.125f : -INFINITY;
        mx0 = fmaxf(mx0, sc[j][e]);
        mx1 = fmaxf(mx1, sc[j][2 + e]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);       // finite: every tile has a visible key
    const float c0 = __expf(m0 - n0), c1 = __expf(m1 - n1);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[j][e] = __expf(sc[j][e] - n0);
        sc[j][2 + e] = __expf(sc[j][2 + e] - n1);
        s0 += sc[j][e];
        s1 += sc[j][2 + e];
      }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    l0 = l0 * c0 + s0;
    l1 = l1 * c1 + s1;
    m0 = n0;
    m1 = n1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[j][0] *= c0; acc[j][1] *= c0;
      acc[j][2] *= c1; acc[j][3] *= c1;
    }
    // ---- O += P V (P as bf16 A fragments; key step s covers key tiles 2s, 2s + 1)
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t pa[4];
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const float* src = sc[2 * s + (hh >> 1)] + ((hh & 1) ? 2 : 0);
        pa[hh] = pack_bf16(src[0], src[1]);
      }
#pragma unroll
      for (int j2 = 0; j2 < 8; j2 += 2) {
        const int mtx = lane >> 3, rr = lane & 7;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + kv_off<true>(16 * s + rr + ((mtx & 1) ? 8 : 0), j2 + (mtx >> 1)), b0, b1, b2, b3);
        mma_bf16_16816(acc[j2], pa, b0, b1);
        mma_bf16_16816(acc[j2 + 1], pa, b2, b3);
      }
    }
    __syncthreads();                    // every warp is done with this stage before it is refilled
  }
  if (failed >= 0) {
    // copies still in flight (this tile's, and the next one's if issued) land before exit (bounded)
    if (threadIdx.x == 0) {
      atomicOr(status, WS_ST_TIMEOUT);
      ea_wait(&bar[failed & 1], (uint32_t)((failed >> 1) & 1));
      if (failed + 1 < n_tiles) ea_wait(&bar[(failed + 1) & 1], (uint32_t)(((failed + 1) >> 1) & 1));
    }
    return;
  }
  const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int col = h * WS_DH + 8 * j + 2 * c;
    if (g < nrows)
      *reinterpret_cast<uint32_t*>(out + (size_t)(row0 + q0 + g) * d + col) = pack_bf16(acc[j][0] * i0, acc[j][1] * i0);
    if (g + 8 < nrows)
      *reinterpret_cast<uint32_t*>(out + (size_t)(row0 + q0 + g + 8) * d + col) =
          pack_bf16(acc[j][2] * i1, acc[j][3] * i1);
  }
}

// ------------------------------------------------------------------ attention on tcgen05
// The same attention with both products on the 5th-generation tensor cores:
// one CTA per (128 query rows, head, window), key tiles of 64; two CTAs
// share an SM.
//   warp 0      TMA producer of Q (once) and the K tiles (three stages);
//   warp 6      TMA producer of the V tiles (two stages) and V transposer:
//               V[key][dim] -> Vt[dim][key] in shared memory (ldmatrix /
//               stmatrix.trans), so both products take K-major operands;
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM buffers,
//               then O += P_{j-1} V_{j-1} (O stays in TMEM);
//   warps 2..5  softmax, one thread per query row (TMEM lane): S_j by
//               tcgen05.ld, scores in log2 units (x log2(e) / 8), running
//               max m, p = 2^(s - m) written as bf16 to P_j (shared memory,
//               the 128-byte-swizzled K-major layout), running sum l of the
//               fp32 weights (their bf16 rounding moves a row's output by
//               ~2^-9 relative at most).  The
//               max m moves only when a row's max grows by more than 8
//               (p stays <= 256); then O is rescaled in TMEM (tcgen05.ld /
//               st) after the previous P V has finished.  At the end
//               O / l is stored as bf16.
// Keys past the window are masked (p = 0).  Every wait is bounded and an
// abort flag in shared memory ends every role's loop after a timeout.
constexpr int FA_Q = 128, FA_K = 64;
constexpr int FA_TILE = FA_K * WS_DH * 2;                 // one 64 x 64 bf16 tile, 8 KB
// shared memory: Q 16 KB | K x3 | V x2 | Vt x2 (8 KB each) | P x2 (16 KB each).
// K tiles are the critical operand (S waits for them), so they get three
// stages and a producer of their own.
constexpr int FA_NK = 3, FA_NV = 2, FA_NVT = 2;
constexpr int FA_THREADS = 224;                           // K producer, MMA, 4 softmax, V producer + transposer
constexpr int FA_OFF_K = 2 * FA_TILE, FA_OFF_V = FA_OFF_K + FA_NK * FA_TILE, FA_OFF_VT = FA_OFF_V + FA_NV * FA_TILE;
constexpr int FA_OFF_P = FA_OFF_VT + FA_NVT * FA_TILE;
constexpr int FA_SMEM = FA_OFF_P + 2 * FA_Q * FA_K * 2 + 1024;
constexpr uint32_t FA_TMEM_COLS = 256;                    // S0 | S1 | O
constexpr uint32_t FA_IDESC = tc::idesc_bf16(FA_Q, FA_K);  // M 128, N 64 (both products)
constexpr float FA_SCALE = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) in log2 units
constexpr float FA_HOLD = 8.0f;                           // max growth (log2) before O is rescaled

struct FaBars {
  uint64_t q_full, k_full[FA_NK], k_empty[FA_NK], v_full[FA_NV], vt_full[FA_NVT], vt_empty[FA_NVT], s_full[2],
      s_empty[2], p_full[2], pv_done[2];
};

__device__ __forceinline__ float fa_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool fa_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > tc::WAIT_BUDGET) {
      *abort = 1;
      atomicOr(status, WS_ST_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform form: lane 0 waits, the warp takes its answer.
__device__ __forceinline__ bool fa_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = fa_wait(bar, parity, abort, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void fa_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// 64 consecutive TMEM columns of this warp's 32 lanes (one wait).
__device__ __forceinline__ void fa_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[16 * q + 0]), "=r"(r[16 * q + 1]), "=r"(r[16 * q + 2]), "=r"(r[16 * q + 3]), "=r"(r[16 * q + 4]),
          "=r"(r[16 * q + 5]), "=r"(r[16 * q + 6]), "=r"(r[16 * q + 7]), "=r"(r[16 * q + 8]), "=r"(r[16 * q + 9]),
          "=r"(r[16 * q + 10]), "=r"(r[16 * q + 11]), "=r"(r[16 * q + 12]), "=r"(r[16 * q + 13]),
          "=r"(r[16 * q + 14]), "=r"(r[16 * q + 15])
        : "r"(taddr + 16u * q));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void fa_st64(uint32_t taddr, const float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr + 16u * q), "r"(__float_as_uint(v[16 * q + 0])), "r"(__float_as_uint(v[16 * q + 1])),
          "r"(__float_as_uint(v[16 * q + 2])), "r"(__float_as_uint(v[16 * q + 3])),
          "r"(__float_as_uint(v[16 * q + 4])), "r"(__float_as_uint(v[16 * q + 5])),
          "r"(__float_as_uint(v[16 * q + 6])), "r"(__float_as_uint(v[16 * q + 7])),
          "r"(__float_as_uint(v[16 * q + 8])), "r"(__float_as_uint(v[16 * q + 9])),
          "r"(__float_as_uint(v[16 * q + 10])), "r"(__float_as_uint(v[16 * q + 11])),
          "r"(__float_as_uint(v[16 * q + 12])), "r"(__float_as_uint(v[16 * q + 13])),
          "r"(__float_as_uint(v[16 * q + 14])), "r"(__float_as_uint(v[16 * q + 15]))
        : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(FA_THREADS, 2) enc_fa_kernel(const __grid_constant__ CUtensorMap tmQKV, bf16* out, int F,
                                                        int d, int32_t* status) {
  extern __shared__ uint8_t fa_dsm[];
  __shared__ __align__(8) FaBars B;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  __shared__ int k_issued[FA_NK], v_issued[FA_NV];   // K / V tile copies requested per stage
  __shared__ int s_commits[2], pv_commits[2];   // S and P V products issued per TMEM / P buffer
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fa_dsm) + 1023) & ~uintptr_t(1023));
  const int qt = blockIdx.x, h = blockIdx.y, i = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = i * F, q0 = qt * FA_Q;
  const int nt = (F + FA_K - 1) / FA_K;
  const int xq = h * WS_DH, xk = d + h * WS_DH, xv = 2 * d + h * WS_DH;
  volatile int* abort = &s_abort;
  if (threadIdx.x == 0) {
    tc::mbar_init(&B.q_full, 1);
    for (int b = 0; b < FA_NK; ++b) { tc::mbar_init(&B.k_full[b], 1); tc::mbar_init(&B.k_empty[b], 1); k_issued[b] = 0; }
    for (int b = 0; b < FA_NV; ++b) { tc::mbar_init(&B.v_full[b], 1); v_issued[b] = 0; }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&B.s_full[b], 1);
      tc::mbar_init(&B.s_empty[b], 4); tc::mbar_init(&B.p_full[b], 4); tc::mbar_init(&B.pv_done[b], 1);
    }
    for (int b = 0; b < FA_NVT; ++b) { tc::mbar_init(&B.vt_full[b], 1); tc::mbar_init(&B.vt_empty[b], 1); }
    s_abort = 0;
    s_commits[0] = s_commits[1] = pv_commits[0] = pv_commits[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::tma_prefetch_desc(&tmQKV);
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, FA_TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  uint8_t* sQ = sm;
  auto sK = [&](int b) { return sm + FA_OFF_K + b * FA_TILE; };
  auto sV = [&](int b) { return sm + FA_OFF_V + b * FA_TILE; };
  auto sVt = [&](int b) { return sm + FA_OFF_VT + b * FA_TILE; };
  auto sP = [&](int b) { return sm + FA_OFF_P + b * (FA_Q * FA_K * 2); };

  if (warp == 0) {
    // ---- Q and K producer (one lane): K tile j waits only for S_{j-3}
    if (lane == 0) {
      tc::mbar_expect_tx(&B.q_full, 2 * FA_TILE);
      tc::tma_load_2d(sQ, &tmQKV, &B.q_full, xq, row0 + q0);
      tc::tma_load_2d(sQ + FA_TILE, &tmQKV, &B.q_full, xq, row0 + q0 + 64);
      for (int j = 0; j < nt; ++j) {
        const int kb = j % FA_NK;
        if (j >= FA_NK && !fa_wait(&B.k_empty[kb], (uint32_t)(((j / FA_NK) & 1) ^ 1), abort, status)) break;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::mbar_expect_tx(&B.k_full[kb], FA_TILE);
        tc::tma_load_2d(sK(kb), &tmQKV, &B.k_full[kb], xk, row0 + j * FA_K);
        ++k_issued[kb];
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ---- V producer and transposer: V tile j + 2 refills the stage of V_j
    // once V_j is transposed; V_j waits for the Vt buffer of P V_{j-2}
    auto load_v = [&](int j) {
      const int b = j % FA_NV;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the transposer's reads of the stage first
      tc::mbar_expect_tx(&B.v_full[b], FA_TILE);
      tc::tma_load_2d(sV(b), &tmQKV, &B.v_full[b], xv, row0 + j * FA_K);
      ++v_issued[b];
    };
    if (lane == 0)
      for (int j = 0; j < FA_NV && j < nt; ++j) load_v(j);
    __syncwarp();
    for (int j = 0; j < nt; ++j) {
      const int b = j % FA_NV, bt = j % FA_NVT;
      if (!fa_wait_warp(&B.v_full[b], (uint32_t)((j / FA_NV) & 1), abort, status)) break;
      if (j >= FA_NVT && !fa_wait_warp(&B.vt_empty[bt], (uint32_t)(((j / FA_NVT) & 1) ^ 1), abort, status)) break;
      // transpose by 8 x 8 blocks: ldmatrix.x4 reads four blocks of V (rows =
      // keys), stmatrix.x4.trans writes them as rows of Vt (rows = head dims)
      const uint32_t vsrc = tc::smem_u32(sV(b)), vdst = tc::smem_u32(sVt(bt));
      const int qm = lane >> 3, r = lane & 7;
#pragma unroll 4
      for (int it = 0; it < 16; ++it) {
        const int blk = it * 4 + qm, kb = blk >> 3, cc = blk & 7;    // key block kb, dim chunk cc
        uint32_t t0, t1, t2, t3;
        ldsm_x4(vsrc + (uint32_t)((kb * 8 + r) * 128 + ((cc ^ r) << 4)), t0, t1, t2, t3);
        const int n = cc * 8 + r;                                    // Vt row (head dim) this lane addresses
        const uint32_t dst = vdst + (uint32_t)(n * 128 + ((kb ^ (n & 7)) << 4));
        asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};"
                     ::"r"(dst), "r"(t0), "r"(t1), "r"(t2), "r"(t3) : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");      // Vt visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        fa_arrive(&B.vt_full[bt]);
        if (j + FA_NV < nt) load_v(j + FA_NV);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint64_t qd = tc::sdesc_sw128(tc::smem_u32(sQ));
      bool ok = fa_wait(&B.q_full, 0, abort, status);
      auto issue_s = [&](int j) -> bool {
        const int b = j & 1, kb = j % FA_NK;
        const uint32_t ph = (uint32_t)((j >> 1) & 1);
        if (!fa_wait(&B.k_full[kb], (uint32_t)((j / FA_NK) & 1), abort, status)) return false;
        if (j >= 2 && !fa_wait(&B.s_empty[b], ph ^ 1u, abort, status)) return false;   // S_{j-2} read
        tc::tc_fence_after();
        const uint64_t kd = tc::sdesc_sw128(tc::smem_u32(sK(kb)));
#pragma unroll
        for (int kk = 0; kk < WS_DH / 16; ++kk)
          tc::umma_bf16(tmem + (uint32_t)(b * FA_K), qd + (uint64_t)(kk * 2), kd + (uint64_t)(kk * 2), FA_IDESC,
                        kk ? 1u : 0u);
        tc::umma_commit(&B.s_full[b]);
        tc::umma_commit(&B.k_empty[kb]);
        ++s_commits[b];
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nt && ok; ++j) {
        if (j + 1 < nt && !issue_s(j + 1)) break;
        const int b = j & 1;
        const uint32_t ph = (uint32_t)((j >> 1) & 1);
        const int bt = j % FA_NVT;
        if (!fa_wait(&B.p_full[b], ph, abort, status) ||
            !fa_wait(&B.vt_full[bt], (uint32_t)((j / FA_NVT) & 1), abort, status))
          break;
        tc::tc_fence_after();
        const uint64_t pd = tc::sdesc_sw128(tc::smem_u32(sP(b))), vd = tc::sdesc_sw128(tc::smem_u32(sVt(bt)));
#pragma unroll
        for (int kk = 0; kk < FA_K / 16; ++kk)
          tc::umma_bf16(tmem + 128u, pd + (uint64_t)(kk * 2), vd + (uint64_t)(kk * 2), FA_IDESC, (j | kk) ? 1u : 0u);
        tc::umma_commit(&B.pv_done[b]);
        tc::umma_commit(&B.vt_empty[bt]);
        ++pv_commits[b];
      }
    }
    __syncwarp();
  } else {
    // ---- softmax: warp w owns TMEM lanes 32 (w % 4) .. + 31
    const int quarter = warp & 3, row = quarter * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1;
      const uint32_t ph = (uint32_t)((j >> 1) & 1);
      if (!fa_wait_warp(&B.s_full[b], ph, abort, status)) { ok = false; break; }
      tc::tc_fence_after();
      float sv[64];
      fa_ld64(tl + (uint32_t)(b * FA_K), sv);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) fa_arrive(&B.s_empty[b]);
      const int nvis = min(FA_K, F - j * FA_K);
      if (nvis < FA_K) {                                         // the window's last tile
#pragma unroll
        for (int k = 0; k < 64; ++k) sv[k] = k < nvis ? sv[k] : -INFINITY;
      }
      // row max of the raw scores: eight independent chains
      float mx8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mx8[q] = sv[q];
#pragma unroll
      for (int k = 8; k < 64; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], sv[k]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * FA_SCALE;
      // the running max moves on the first tile, or when it grew by more than FA_HOLD
      const bool move = j == 0 || mx > m + FA_HOLD;
      const float mnew = move ? fmaxf(m, mx) : m;
      const float alpha = (j == 0) ? 0.0f : fa_ex2(m - mnew);    // 1 when the max stays
      m = mnew;
      // p = 2^(s * scale - m): one FFMA and one EX2 per score; eight partial sums
      float sum8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) sum8[q] = 0.0f;
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        const float p0 = fa_ex2(fmaf(sv[k], FA_SCALE, -m)), p1 = fa_ex2(fmaf(sv[k + 1], FA_SCALE, -m));
        sum8[(k >> 1) & 7] += p0 + p1;
        pk[k / 2] = pack_bf16(p0, p1);
      }
      const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      l = l * alpha + sum;
      // P_j's buffer was last read by P V of tile j - 2
      if (j >= 2 && !fa_wait_warp(&B.pv_done[b], ph ^ 1u, abort, status)) { ok = false; break; }
      if (j >= 1 && __any_sync(0xffffffffu, move)) {
        // rescale O: its last update (P V of tile j - 1) must be complete
        if (!fa_wait_warp(&B.pv_done[b ^ 1], (uint32_t)(((j - 1) >> 1) & 1), abort, status)) { ok = false; break; }
        tc::tc_fence_after();
        float ov[64];
        fa_ld64(tl + 128u, ov);
#pragma unroll
        for (int c = 0; c < 64; ++c) ov[c] *= alpha;
        fa_st64(tl + 128u, ov);
      }
      uint8_t* prow = sP(b) + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) fa_arrive(&B.p_full[b]);
    }
    if (ok) {
      const int jl = nt - 1;
      ok = fa_wait_warp(&B.pv_done[jl & 1], (uint32_t)((jl >> 1) & 1), abort, status);
    }
    if (ok) {
      tc::tc_fence_after();
      float ov[64];
      fa_ld64(tl + 128u, ov);
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      if (q0 + row < F) {
        uint4* dst = reinterpret_cast<uint4*>(out + (size_t)(row0 + q0 + row) * d + h * WS_DH);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float* o8 = ov + 8 * c;
          dst[c] = make_uint4(pack_bf16(o8[0] * inv, o8[1] * inv), pack_bf16(o8[2] * inv, o8[3] * inv),
                              pack_bf16(o8[4] * inv, o8[5] * inv), pack_bf16(o8[6] * inv, o8[7] * inv));
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) {
    // after a timeout: copies requested and products issued complete (bounded) before the CTA exits
    for (int b = 0; b < FA_NK; ++b)
      if (k_issued[b] > 0) tc::mbar_wait(&B.k_full[b], (uint32_t)((k_issued[b] - 1) & 1));
    for (int b = 0; b < FA_NV; ++b)
      if (v_issued[b] > 0) tc::mbar_wait(&B.v_full[b], (uint32_t)((v_issued[b] - 1) & 1));
    for (int b = 0; b < 2; ++b) {
      if (s_commits[b] > 0) tc::mbar_wait(&B.s_full[b], (uint32_t)((s_commits[b] - 1) & 1));
      if (pv_commits[b] > 0) tc::mbar_wait(&B.pv_done[b], (uint32_t)((pv_commits[b] - 1) & 1));
    }
    tc::mbar_wait(&B.q_full, 0);
  }
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, FA_TMEM_COLS);
}

// ------------------------------------------------------------------ host helpers
const TcMap* act_map(ws_enc* e, const void* base, int rows, int cols, int bn) {
  auto key = std::make_tuple(base, rows, bn);
  auto it = e->maps.find(key);
  if (it != e->maps.end()) return &it->second;
  TcMap m;
  if (!tc_encode_map(&m, base, (uint64_t)rows, (uint64_t)cols, (uint32_t)bn)) return nullptr;
  return &e->maps.emplace(key, m).first->second;
}

cudaError_t enc_gemm(ws_enc* e, const void* X, int M, const bf16* W, const TcMap& mw, int N, int K, const Epi& ep,
                     cudaStream_t s) {
  GemmShape g;
  g.X = X; g.ldx = K; g.W = W; g.ldw = K; g.M = M; g.N = N; g.K = K; g.batch = 1;
  const TcMap* mx = act_map(e, X, M, K, tc_pick_bn(M, N, 1));
  if (!mx) return cudaErrorInvalidValue;
  return launch_gemm_tc(g, ep, mw, mx, X, (uint64_t)M, 1, s, false);
}

Epi epi_of(ws_enc* e, int kind) {
  Epi ep;
  memset(&ep, 0, sizeof ep);
  ep.kind = kind;
  ep.d = e->d.d_model;
  ep.status = e->status;
  return ep;
}

}  // namespace

extern "C" {

size_t ws_encoder_workspace(const ws_encoder_desc* desc) {
  if (check_enc_desc(desc)) return 0;
  return plan(*desc).total;
}

int ws_encoder_load(ws_enc** out, const ws_encoder_desc* desc, void* workspace, size_t bytes, const void* blob,
                    ws_stream stream) {
  ws_enc* e = nullptr;
  if (!out) return efail(nullptr, WS_EINVAL, "null output handle");
  *out = nullptr;
  if (const char* m = check_enc_desc(desc)) return efail(nullptr, WS_EINVAL, "%s", m);
  if (!workspace || !blob) return efail(nullptr, WS_EINVAL, "null workspace or blob");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return efail(nullptr, WS_EINVAL, "workspace must be 256-byte aligned");
  const EncPlan p = plan(*desc);
  if (bytes < p.total) return efail(nullptr, WS_ENOSPACE, "workspace %zu < %zu bytes", bytes, p.total);
  if (!tc_engine_available()) return efail(nullptr, WS_EUNSUPPORTED, "the encoder needs the tcgen05 engine (TMA)");
  e = new ws_enc;
  e->d = *desc;
  const ws_encoder_desc& d = e->d;
  const int D = d.d_model, Fd = d.d_ff;
  e->kp = (3 * d.n_mels + 63) / 64 * 64;
  char* b = static_cast<char*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;
  auto bail = [&](int code) { *out = nullptr; ws_enc* tmp = e; g_enc_err = tmp->err; delete tmp; return code; };
  cudaError_t r = cudaMemcpyAsync(b + p.blob, blob, blob_elems(d) * 2, cudaMemcpyDefault, s);
  if (r != cudaSuccess) { efail(e, WS_ECUDA, "blob copy: %s", cudaGetErrorString(r)); return bail(WS_ECUDA); }
  const bf16* w = reinterpret_cast<const bf16*>(b + p.blob);
  auto take = [&](size_t n) { const bf16* q = w; w += n; return q; };
  const bf16* conv1_w = take((size_t)D * d.n_mels * 3);
  e->b1 = take(D);
  const bf16* conv2_w = take((size_t)D * D * 3);
  e->b2 = take(D);
  e->layers.resize(d.n_layers);
  std::vector<const bf16*> bq(d.n_layers), bv(d.n_layers);
  for (int l = 0; l < d.n_layers; ++l) {
    EncLayer& L = e->layers[l];
    L.ln1_g = take(D); L.ln1_b = take(D);
    L.w_qkv = take((size_t)3 * D * D); bq[l] = take(D); bv[l] = take(D);
    L.w_o = take((size_t)D * D); L.b_o = take(D);
    L.ln2_g = take(D); L.ln2_b = take(D);
    L.w_fc1 = take((size_t)Fd * D); L.b_fc1 = take(Fd);
    L.w_fc2 = take((size_t)D * Fd); L.b_fc2 = take(D);
    L.b_qkv = reinterpret_cast<bf16*>(b + p.bqkv) + (size_t)l * 3 * D;
  }
  e->lnp_g = take(D); e->lnp_b = take(D);
  e->w1 = reinterpret_cast<bf16*>(b + p.w1);
  e->w2 = reinterpret_cast<bf16*>(b + p.w2);
  e->pos = reinterpret_cast<float*>(b + p.pos);
  e->x1 = reinterpret_cast<bf16*>(b + p.x1);
  e->h1 = reinterpret_cast<bf16*>(b + p.h1);
  e->x2 = reinterpret_cast<bf16*>(b + p.x2);
  e->x = reinterpret_cast<float*>(b + p.x);
  e->h = reinterpret_cast<bf16*>(b + p.h);
  e->qkv = reinterpret_cast<bf16*>(b + p.qkv);
  e->ao = reinterpret_cast<bf16*>(b + p.ao);
  e->ffn = reinterpret_cast<bf16*>(b + p.ffn);
  e->status = reinterpret_cast<int32_t*>(b + p.status);
  // repacked convolutions, assembled q|k|v biases, the position table
  if (r == cudaSuccess) {
    cudaLaunchConfig_t c1 = cfg_of(dim3(1024), dim3(256), 0, s);
    r = cudaLaunchKernelEx(&c1, conv_repack_kernel, conv1_w, e->w1, D, d.n_mels, e->kp);
  }
  if (r == cudaSuccess) {
    cudaLaunchConfig_t c2 = cfg_of(dim3(1024), dim3(256), 0, s);
    r = cudaLaunchKernelEx(&c2, conv_repack_kernel, conv2_w, e->w2, D, D, 3 * D);
  }
  for (int l = 0; l < d.n_layers && r == cudaSuccess; ++l) {
    cudaLaunchConfig_t c3 = cfg_of(dim3(8), dim3(256), 0, s);
    r = cudaLaunchKernelEx(&c3, qkv_bias_kernel, bq[l], bv[l], e->layers[l].b_qkv, D);
  }
  if (r == cudaSuccess) {
    cudaLaunchConfig_t c4 = cfg_of(dim3(512), dim3(256), 0, s);
    r = cudaLaunchKernelEx(&c4, enc_pos_table_kernel, e->pos, d.n_frames, D);
  }
  if (r == cudaSuccess) r = cudaMemsetAsync(e->status, 0, 4, s);
  if (r == cudaSuccess) r = cudaStreamSynchronize(s);
  if (r != cudaSuccess) { efail(e, WS_ECUDA, "encoder set-up: %s", cudaGetErrorString(r)); return bail(WS_ECUDA); }
  ws_count_launches(3 + d.n_layers);
  bool ok = tc_encode_map(&e->m_w1, e->w1, (uint64_t)D, (uint64_t)e->kp, 128) &&
            tc_encode_map(&e->m_w2, e->w2, (uint64_t)D, (uint64_t)3 * D, 128);
  for (auto& L : e->layers) {
    ok = ok && tc_encode_map(&L.m_qkv, L.w_qkv, (uint64_t)3 * D, (uint64_t)D, 128);
    ok = ok && tc_encode_map(&L.m_o, L.w_o, (uint64_t)D, (uint64_t)D, 128);
    ok = ok && tc_encode_map(&L.m_fc1, L.w_fc1, (uint64_t)Fd, (uint64_t)D, 128);
    ok = ok && tc_encode_map(&L.m_fc2, L.w_fc2, (uint64_t)D, (uint64_t)Fd, 128);
  }
  if (!ok) { efail(e, WS_ECUDA, "tensor map encoding failed"); return bail(WS_ECUDA); }
  r = tc_init_attributes();
  if (r == cudaSuccess) r = cudaFuncSetAttribute(enc_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, EA_SMEM);
  if (r == cudaSuccess) r = cudaFuncSetAttribute(enc_fa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FA_SMEM);
  if (r != cudaSuccess) { efail(e, WS_ECUDA, "kernel attributes: %s", cudaGetErrorString(r)); return bail(WS_ECUDA); }
  *out = e;
  return WS_OK;
}

int ws_encode(ws_enc* e, int n, const void* mel, void* out, ws_stream stream) {
  if (!e) return efail(nullptr, WS_EINVAL, "null encoder");
  if (n < 0 || n > e->d.max_batch) return efail(e, WS_EINVAL, "n %d outside 0..max_batch (%d)", n, e->d.max_batch);
  if (n == 0) return WS_OK;
  if (!mel || !out) return efail(e, WS_EINVAL, "null mel or out");
  const ws_encoder_desc& d = e->d;
  const int D = d.d_model, Fd = d.d_ff, F = d.n_frames, T = 2 * F;
  const int M1 = n * T, M = n * F;
  cudaStream_t s = (cudaStream_t)stream;
  cudaLaunchConfig_t c;
  // ---- stem: conv1 (im2col GEMM + GELU), conv2 (im2col GEMM + GELU), + positions
  c = cfg_of(dim3(M1), dim3(128), 0, s);
  ECK(cudaLaunchKernelEx(&c, im2col1_kernel, (const bf16*)mel, e->x1, d.n_mels, T, e->kp));
  Epi ep = epi_of(e, EPI_GELU);
  ep.bias = e->b1; ep.out = e->h1; ep.ldo = D;
  ECK(enc_gemm(e, e->x1, M1, e->w1, e->m_w1, D, e->kp, ep, s));
  c = cfg_of(dim3(M), dim3(128), 0, s);
  ECK(cudaLaunchKernelEx(&c, im2col2_kernel, (const bf16*)e->h1, e->x2, D, F));
  ep = epi_of(e, EPI_GELU);
  ep.bias = e->b2; ep.out = e->h; ep.ldo = D;
  ECK(enc_gemm(e, e->x2, M, e->w2, e->m_w2, D, 3 * D, ep, s));
  c = cfg_of(dim3(1216), dim3(256), 0, s);
  ECK(cudaLaunchKernelEx(&c, add_pos_kernel, (const bf16*)e->h, (const float*)e->pos, e->x, D, F, (size_t)M * D));
  ws_count_launches(3);
  // ---- blocks
  const TcMap* mq = act_map(e, e->qkv, M, 3 * D, WS_XCHUNK);
  if (!mq) return efail(e, WS_ECUDA, "QKV tensor map");
  const int qtiles = (F + 63) / 64;
  for (int l = 0; l < d.n_layers; ++l) {
    const EncLayer& L = e->layers[l];
    ECK(launch_layernorm<bf16>(M, D, e->x, D, L.ln1_g, L.ln1_b, e->h, D, 0, s, false));
    ep = epi_of(e, EPI_STORE);
    ep.bias = L.b_qkv; ep.out = e->qkv; ep.ldo = 3 * D;
    ECK(enc_gemm(e, e->h, M, L.w_qkv, L.m_qkv, 3 * D, D, ep, s));
    if (e->attn_tc) {
      c = cfg_of(dim3((F + FA_Q - 1) / FA_Q, D / WS_DH, n), dim3(FA_THREADS), FA_SMEM, s);
      ECK(cudaLaunchKernelEx(&c, enc_fa_kernel, *reinterpret_cast<const CUtensorMap*>(mq), e->ao, F, D, e->status));
    } else {
      c = cfg_of(dim3(qtiles, D / WS_DH, n), dim3(128), EA_SMEM, s);
      ECK(cudaLaunchKernelEx(&c, enc_attn_kernel, *reinterpret_cast<const CUtensorMap*>(mq), (const bf16*)e->qkv,
                             e->ao, F, D, e->status));
    }
    ws_count_launches(1);
    ep = epi_of(e, EPI_RESID);
    ep.bias = L.b_o; ep.resid = e->x; ep.ldr = D;
    ECK(enc_gemm(e, e->ao, M, L.w_o, L.m_o, D, D, ep, s));
    ECK(launch_layernorm<bf16>(M, D, e->x, D, L.ln2_g, L.ln2_b, e->h, D, 0, s, false));
    ep = epi_of(e, EPI_GELU);
    ep.bias = L.b_fc1; ep.out = e->ffn; ep.ldo = Fd;
    ECK(enc_gemm(e, e->h, M, L.w_fc1, L.m_fc1, Fd, D, ep, s));
    ep = epi_of(e, EPI_RESID);
    ep.bias = L.b_fc2; ep.resid = e->x; ep.ldr = D;
    ECK(enc_gemm(e, e->ffn, M, L.w_fc2, L.m_fc2, D, Fd, ep, s));
  }
  ECK(launch_layernorm<bf16>(M, D, e->x, D, e->lnp_g, e->lnp_b, (bf16*)out, D, 0, s, false));
  return WS_OK;
}

int ws_encoder_status(ws_enc* e, ws_stream stream, int32_t* host_status) {
  if (!e) return efail(nullptr, WS_EINVAL, "null encoder");
  cudaStream_t s = (cudaStream_t)stream;
  int32_t v = 0;
  ECK(cudaMemcpyAsync(&v, e->status, 4, cudaMemcpyDeviceToHost, s));
  ECK(cudaStreamSynchronize(s));
  ECK(cudaMemsetAsync(e->status, 0, 4, s));
  ECK(cudaStreamSynchronize(s));
  if (host_status) *host_status = v;
  if (v) return efail(e, WS_EDEVICE, "device status 0x%x (8 = a bounded wait ran out)", v);
  return WS_OK;
}

int ws_encoder_attention(ws_enc* e, int mode) {
  if (!e) return efail(nullptr, WS_EINVAL, "null encoder");
  if (mode == 0 || mode == 1) e->attn_tc = mode;
  return e->attn_tc;
}

const char* ws_encoder_error(const ws_enc* e) { return e ? e->err.c_str() : g_enc_err.c_str(); }

void ws_encoder_free(ws_enc* e) { delete e; }

}  // extern "C"
