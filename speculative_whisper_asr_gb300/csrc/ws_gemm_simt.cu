// SIMT GEMM engine: Y = X W^T with a fused epilogue, fp32 FMA on CUDA cores.
//
// Used for the fp32 model (the tensor cores' tf32 would not hold the fp32
// tolerance) and as the reference GPU engine for bf16.  Every output element
// is one thread's sequential fmaf chain over k = 0..K-1, so its value does
// not depend on M, on the tile it falls in, or on the launch shape: a row
// verified inside a 9-row block equals the same row decoded alone.
#include "ws_epilogue.cuh"

namespace {

constexpr int BF = 64;   // features per CTA
constexpr int KC = 32;   // k per smem stage

template <typename T, int BT>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmShape g, Epi e) {
  __shared__ float Ws[BF][KC + 1];
  __shared__ float Xs[BT][KC + 1];
  constexpr int TT = BT / 16;            // tokens per thread
  const int tid = threadIdx.x;
  const int fq = tid & 15, tq = tid >> 4;
  const int f0 = blockIdx.x * BF, t0 = blockIdx.y * BT, z = blockIdx.z;
  const T* W = reinterpret_cast<const T*>(g.W);
  const T* X = reinterpret_cast<const T*>(g.X);
  int M = g.M;
  pdl_wait();
  if (e.kind == EPI_CROSSKV) {
    int a = e.cu_frames[z], b = e.cu_frames[z + 1];
    X += (size_t)a * g.ldx;
    M = min(b - a, e.xkv.max_frames);
  }
  if (t0 >= M) { pdl_trigger(); return; }

  float acc[4][TT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < TT; ++j) acc[i][j] = 0.0f;

  const int N = g.N, K = g.K;
  for (int k0 = 0; k0 < K; k0 += KC) {
    {
      const int row = tid >> 2, seg = (tid & 3) * 8, f = f0 + row;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        int k = k0 + seg + u;
        Ws[row][seg + u] = (f < N && k < K) ? to_f<T>(W[(size_t)f * g.ldw + k]) : 0.0f;
      }
    }
    for (int idx = tid; idx < BT * KC; idx += 256) {
      int row = idx / KC, kk = idx - row * KC, t = t0 + row, k = k0 + kk;
      Xs[row][kk] = (t < M && k < K) ? to_f<T>(X[(size_t)t * g.ldx + k]) : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < KC; ++kk) {
      float w[4], x[TT];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = Ws[fq * 4 + i][kk];
#pragma unroll
      for (int j = 0; j < TT; ++j) x[j] = Xs[tq * TT + j][kk];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < TT; ++j) acc[i][j] = fmaf(w[i], x[j], acc[i][j]);
    }
    __syncthreads();
  }
  pdl_trigger();

  if (e.kind == EPI_LOGITS) {
#pragma unroll
    for (int j = 0; j < TT; ++j) {
      int t = t0 + tq * TT + j;
      unsigned long long best = 0ull;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        int n = f0 + fq * 4 + i;
        if (n < N && t < M) {
          float v = epi_logit(e, n, acc[i][j]);
          if (e.logits) e.logits[(long long)t * e.ldl + n] = v;
          unsigned long long key = argmax_key(v, n);
          best = key > best ? key : best;
        }
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      if (fq == 0 && t < M && e.amax) atomicMax(e.amax + t, best);
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < TT; ++j) {
    int t = t0 + tq * TT + j;
    if (t >= M) continue;
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
      int n = f0 + fq * 4 + i;
      if (n < N) epi_pair<T>(e, t, n, acc[i][j], acc[i + 1][j], z);
    }
  }
}

template <typename T, int BT>
cudaError_t launch_bt(const GemmShape& g, const Epi& e, cudaStream_t s, bool pdl) {
  dim3 grid((g.N + BF - 1) / BF, (g.M + BT - 1) / BT, g.batch > 0 ? g.batch : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  ws_count_launches(1);
  return cudaLaunchKernelEx(&cfg, gemm_simt_kernel<T, BT>, g, e);
}

}  // namespace

template <typename T>
cudaError_t launch_gemm_simt(const GemmShape& g, const Epi& e, cudaStream_t s, bool pdl) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  if (g.M <= 16) return launch_bt<T, 16>(g, e, s, pdl);
  return launch_bt<T, 32>(g, e, s, pdl);
}

template cudaError_t launch_gemm_simt<float>(const GemmShape&, const Epi&, cudaStream_t, bool);
template cudaError_t launch_gemm_simt<bf16>(const GemmShape&, const Epi&, cudaStream_t, bool);
