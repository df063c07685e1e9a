// Persistent block-verification kernel: stage table and call arguments
// (host <-> device).  Internal to libws.
#pragma once
#include "ws_internal.cuh"

#define FUSED_MAX_RING 12    // shared-memory ring slots (16 KB each) at most
#define FUSED_MAX_ROWS 16    // query rows one call may carry

enum FusedKind { FS_EMBED = 0, FS_GEMM = 1, FS_SELF = 2, FS_CROSS = 3, FS_ARGMAX = 4 };
enum FusedIn { FIN_LN = 0, FIN_ACT = 1 };

// One stage of the verify pass.  GEMM stages: Y = In . W^T with W [N, K]
// (TMA map `map`, 128-row boxes), In either LayerNorm(x; ln_g, ln_b) or a
// bf16 activation buffer, split-K factor `splits` (the per-op path's), and
// the epilogue `epi` with its bias / output.
struct FusedStage {
  int kind;
  int layer;
  const void* map;             // CUtensorMap in device memory (64-byte aligned)
  int N, kb_total, splits;
  int in_kind;
  const void* ln_g;
  const void* ln_b;
  const bf16* act;
  int ld_act;
  int epi;
  const void* bias;
  const void* bias2;
  void* out;
  int ldo;
  int hist_idx;                // residual copy into the drafter history (-1: none)
};

struct FusedArgs {
  const FusedStage* stages;
  int n_stages;
  int ring_slots;
  size_t work_bytes;           // shared-memory work region (B operand, attention scratch, split-K fold)
  int n, H, M;                 // requests, rows per request, rows
  int d, V, heads, max_pos, max_block, n_hist;
  int nsplit_self, nsplit_cross;
  RowMap rm;
  const int32_t* req_ids;
  const int32_t* block;        // [n, H]
  const int32_t* block_len;    // [n]
  const bf16* tok_emb;         // [V, d]
  const bf16* pos_emb;         // [max_pos, d]
  float* x;                    // residual [rows, d]
  bf16* ao;                    // attention output [rows, d]
  bf16* q;                     // queries [rows, d]
  char* kv;                    // self K/V pool of layer 0
  size_t kv_layer_bytes;
  const int32_t* ptab;
  int ppr;
  XKV xkv;
  const int32_t* Fv;           // valid frames per slot
  float* hist;
  float* part;                 // split-K partials [tile][split][16][128]
  int* tile_ctr;               // per-tile arrival counters, zero between stages
  float* apart;                // attention partials [rows][heads][splits][66]
  int* actr;                   // attention arrival counters [max_batch][heads]
  unsigned long long* amax;    // [rows] argmax keys
  float* logits;               // [rows, V] or NULL
  const uint32_t* suppress;
  int32_t* target;             // [n, H] out
  int32_t* pend_start;
  int32_t* pend_n;
  unsigned* gbar;              // grid barrier: [0] arrivals, [1] generation
  int32_t* status;
};

// Shared-memory bytes of the work region (B operand or attention scratch)
// for a largest GEMM unit of `max_unit_kb` k-blocks.
size_t fused_work_bytes(int max_unit_kb);
// Configure the kernel (shared-memory limit) and return how many ring slots
// fit beside `work_bytes`; 0 when the device cannot run it (occupancy < 1 CTA/SM).
int fused_prepare(size_t work_bytes, int* grid_ctas);
cudaError_t launch_fused_verify(const FusedArgs& a, int grid, size_t work_bytes, cudaStream_t s);
