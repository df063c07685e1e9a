// Dataflow block verification for one-request contexts: arguments shared by
// the host set-up (ws_api.cu) and the kernel (ws_flow.cu).  Internal to libws.
#pragma once
#include "ws_internal.cuh"

#define FLOW_MAX_ROWS 16       // block rows one call may carry (a 16-token MMA tile)
#define FLOW_CTR_LAYER 512     // dependency counters per decoder layer (ints)
#define FLOW_CTR_GLOBAL 16     // counters after the per-layer blocks
#define FLOW_XS_BYTES 46080    // shared-memory staging of residual rows for a layer norm
#define FLOW_GP 68             // floats per cross-attention group partial (m, l, 64 values, pad)

// Counter offsets inside one layer's block.
enum FlowCtr {
  FC_QKV_HEAD = 0,        // [heads] QKV tasks done per head (12 = q, k, v of 64 features each)
  FC_QC_HEAD = 64,        // [heads] cross-query tasks done per head (4)
  FC_X_ARRIVE = 128,      // [heads] cross-attention chunk groups done per head
  FC_FC1_PIECE = 192,     // [f / d] FC1 tasks done per d-wide slice of the FFN
  FC_SELF_DONE = 200,     // heads whose self-attention output is stored
  FC_O_DONE = 201,        // output-projection tasks done
  FC_X_DONE = 202,        // heads whose cross-attention output is stored
  FC_OC_DONE = 203,       // cross-output-projection tasks done
  FC_FC2_DONE = 204,      // FC2 row tiles folded into the residual
  FC_FC2_ARRIVE = 256     // [d / 16] FC2 k-slices done per row tile
};
enum FlowGlobalCtr { FG_EMBED = 0, FG_HEAD_ARRIVE = 1, FG_EXIT = 2, FG_ABORT = 3 };

// One decoder layer: weight maps (16-row x 64-column boxes, 128-byte
// swizzle; CUtensorMap in device memory), biases and layer-norm parameters.
struct FlowLayer {
  const void* map_qkv;
  const void* map_o;
  const void* map_qc;
  const void* map_oc;
  const void* map_fc1;
  const void* map_fc2;
  const bf16 *b_q, *b_v, *b_o, *b_qc, *b_oc, *b_fc1, *b_fc2;
  const bf16 *ln1_g, *ln1_b, *ln2_g, *ln2_b, *ln3_g, *ln3_b;
  int hist_idx;                // index among the history layers, or -1
};

struct FlowArgs {
  const FlowLayer* layers;     // [n_layers] (device)
  const void* map_head;        // tied LM head (token embedding), 16-row boxes
  const void* map_ao;          // attention output [rows, d], 16-row boxes
  const void* map_ffn;         // FFN activation [rows, f], 16-row boxes
  const void* map_kv;          // self K/V pool as [rows, 64], 64 x 64 boxes
  const void* map_xkv;         // acoustic K/V slabs as [rows, 64], 64 x 64 boxes
  const void* map_x;           // fp32 residual [rows, d], boxes of xs_rows whole rows
  int xs_rows;                 // residual rows one layer-norm staging pass holds
  int n_layers, d, f, heads, V, max_pos, max_block, n_hist;
  int H;                       // block rows of this call (one request)
  const int32_t* req_ids;      // [1]
  const int32_t* block;        // [1, H]
  const int32_t* block_len;    // [1]
  const bf16* tok_emb;
  const bf16* pos_emb;
  const bf16* lnf_g;
  const bf16* lnf_b;
  float* x;                    // residual [rows, d] fp32
  bf16* q;                     // queries [rows, d]
  bf16* ao;                    // attention output [rows, d]
  bf16* ffn;                   // FFN activation [rows, f]
  int32_t* L;
  const int32_t* Fv;
  int32_t* pend_start;
  int32_t* pend_n;
  char* kv;                    // self K/V pool of layer 0 (bytes)
  size_t kv_layer_bytes;
  const int32_t* ptab;
  int ppr;
  size_t xkv_slot_rows, xkv_layer_rows;   // rows of map_xkv per request slot / per layer
  int max_frames;
  float* hist;                 // history residuals [slot][max_block][n_hist][d]
  float* xpart;                // cross-attention group partials [heads][max_groups][16][FLOW_GP]
  int max_groups;              // groups of four 64-frame chunks per head
  float* fpart;                // FC2 partials [d / 16][f / d][16][16]
  unsigned long long* amax;    // [16] argmax keys
  float* logits;               // [H, V] or NULL
  const uint32_t* suppress;
  int32_t* target;             // [1, H]
  int* ctr;                    // [n_layers * FLOW_CTR_LAYER + FLOW_CTR_GLOBAL], zero between launches
  int32_t* status;
};

// Configure the kernel (shared-memory limit) and return the grid (one CTA
// per SM), or 0 when the device cannot co-schedule it.
int flow_prepare();
size_t flow_smem_bytes();
cudaError_t launch_flow_verify(const FlowArgs& a, int grid, cudaStream_t s);
