// Greedy token selection over given logits rows, for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured (allocation is not a capturable operation), code embedded
// in a host framework that owns every byte of device memory through its own
// pool and forbids side allocations, and latency-critical threads where an
// allocation could block on the driver.  They still need the greedy choice
// of Whisper's decoder (argmax over the vocabulary, lowest id on ties) for
// logits they hold.  This entry point does the same reduction as the
// LM-head argmax of ws_verify, but its partial results live in a file-scope
// device array instead of a caller workspace.
//
// Scratch: g_argmax_part holds one partial key per (row, chunk); at most
// WS_NOALLOC_MAX_ROWS rows per call (256 KB, held by every GPU that loads the
// library until the process exits).  Pass 1 writes every entry pass 2 reads,
// so nothing has to start at zero.  All calls share the array: calls whose
// kernels overlap on the GPU (different streams, or different host threads
// without ordering) race and must not be issued.
#include <mutex>
#include <string>

#include "ws_internal.cuh"

#define WS_NOALLOC_MAX_ROWS 1024
#define WS_NOALLOC_CHUNKS 32

static __device__ __align__(256) unsigned long long g_argmax_part[WS_NOALLOC_MAX_ROWS * WS_NOALLOC_CHUNKS];

namespace {

constexpr int NT = 256;

// Pass 1: block (row, chunk) reduces ids [chunk * C, min(V, (chunk + 1) * C)).
__global__ void __launch_bounds__(NT) noalloc_argmax_part(const float* logits, int V, const uint32_t* sup,
                                                          unsigned long long* part) {
  __shared__ unsigned long long sh[NT / 32];
  const int row = blockIdx.x, chunk = blockIdx.y;
  const int C = (V + WS_NOALLOC_CHUNKS - 1) / WS_NOALLOC_CHUNKS;
  const int lo = chunk * C, hi = min(V, lo + C);
  const float* z = logits + (size_t)row * V;
  unsigned long long best = 0ull;
  for (int v = lo + threadIdx.x; v < hi; v += NT) {
    const float y = (sup && ((sup[v >> 5] >> (v & 31)) & 1u)) ? -INFINITY : z[v];
    const unsigned long long k = argmax_key(y, v);
    best = k > best ? k : best;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
    best = other > best ? other : best;
  }
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < NT / 32; ++w) best = sh[w] > best ? sh[w] : best;
    best = sh[0] > best ? sh[0] : best;
    part[(size_t)row * WS_NOALLOC_CHUNKS + chunk] = best;
  }
}

// Pass 2: one thread per row folds the chunk keys.
__global__ void noalloc_argmax_final(int rows, const unsigned long long* part, int32_t* out) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= rows) return;
  unsigned long long best = 0ull;
  for (int c = 0; c < WS_NOALLOC_CHUNKS; ++c) {
    const unsigned long long k = part[(size_t)row * WS_NOALLOC_CHUNKS + c];
    best = k > best ? k : best;
  }
  out[row] = argmax_key_id(best);
}

// Device address of g_argmax_part per CUDA context: a __device__ array has
// its own copy, at its own address, in every context that loads the module
// (the primary context of each device, any context a host framework creates
// itself, a fresh primary context after cudaDeviceReset).  Entries are
// looked up with the context current and never cross contexts.
struct PartAddr {
  void* ctx;
  unsigned long long* ptr;
};
std::mutex g_mu;
PartAddr g_part[64] = {};
int g_n_part = 0;
using CtxGetCurrent = int (*)(void**);     // CUresult cuCtxGetCurrent(CUcontext*)
CtxGetCurrent g_ctx_get = nullptr;

int fail(int code, const char* msg) {
  ws_set_thread_error(msg);   // readable through ws_last_error(NULL)
  return code;
}

// The calling thread's current context (after making sure the runtime has
// one), or nullptr.  Called with g_mu held.
void* current_context() {
  if (!g_ctx_get) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    g_ctx_get = reinterpret_cast<CtxGetCurrent>(fn);
  }
  void* ctx = nullptr;
  if (g_ctx_get(&ctx) != 0) return nullptr;
  if (!ctx) {
    // no context on this thread yet: the runtime binds the device's primary one
    if (cudaFree(nullptr) != cudaSuccess || g_ctx_get(&ctx) != 0) return nullptr;
  }
  return ctx;
}

}  // namespace

extern "C" int ws_argmax_rows_noalloc(const float* logits, int rows, int vocab, const uint32_t* suppress,
                                      int32_t* out, ws_stream stream) {
  if (!logits || !out) return fail(WS_EINVAL, "null logits or output");
  if (rows < 0 || vocab < 1) return fail(WS_EINVAL, "rows must be >= 0 and vocab >= 1");
  if (rows > WS_NOALLOC_MAX_ROWS) return fail(WS_EINVAL, "rows exceed the no-allocation scratch capacity (1024)");
  if (rows == 0) return WS_OK;
  // an error left by the caller's earlier work is reported as such, not as ours
  if (cudaError_t prior = cudaPeekAtLastError(); prior != cudaSuccess)
    return fail(WS_ECUDA, (std::string("a CUDA error was pending before this call: ") +
                           cudaGetErrorString(prior)).c_str());
  unsigned long long* part = nullptr;
  {
    // once per context, with that context current: host code needs the
    // array's device address (its name on the host is only a stand-in)
    std::lock_guard<std::mutex> lk(g_mu);
    void* ctx = current_context();
    if (!ctx) return fail(WS_ECUDA, "no current CUDA context");
    for (int i = 0; i < g_n_part; ++i)
      if (g_part[i].ctx == ctx) part = g_part[i].ptr;
    if (!part) {
      if (g_n_part == 64) return fail(WS_ECUDA, "more than 64 CUDA contexts used this entry point");
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_argmax_part);
      if (e != cudaSuccess || !p) return fail(WS_ECUDA, "cudaGetSymbolAddress of the scratch array failed");
      part = static_cast<unsigned long long*>(p);
      g_part[g_n_part++] = {ctx, part};
    }
  }
  cudaStream_t s = (cudaStream_t)stream;
  void* a1[] = {(void*)&logits, (void*)&vocab, (void*)&suppress, (void*)&part};
  cudaError_t e = cudaLaunchKernel((const void*)noalloc_argmax_part, dim3(rows, WS_NOALLOC_CHUNKS), dim3(NT), a1,
                                   0, s);
  if (e != cudaSuccess) return fail(WS_ECUDA, (std::string("pass 1 launch: ") + cudaGetErrorString(e)).c_str());
  const unsigned long long* cpart = part;
  void* a2[] = {(void*)&rows, (void*)&cpart, (void*)&out};
  e = cudaLaunchKernel((const void*)noalloc_argmax_final, dim3((rows + 127) / 128), dim3(128), a2, 0, s);
  ws_count_launches(e == cudaSuccess ? 2 : 1);
  if (e != cudaSuccess) return fail(WS_ECUDA, (std::string("pass 2 launch: ") + cudaGetErrorString(e)).c_str());
  return WS_OK;
}
