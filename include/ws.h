/*
 * ws.h — C ABI of the speculative Whisper decoding library (libws.so).
 *
 * The library implements the data-parallel hot path of Whisper-Flash
 * ("Whisper-Flash: Acoustically Conditioned Parallel Drafting for Faster
 * Whisper Decoding", arXiv 2609.32869): a two-layer parallel drafter fills
 * K mask positions after the latest token (§3.2, Eq. 2), the frozen target
 * decoder verifies the K+1-token block in one causal pass and keeps the
 * longest prefix matching its own greedy argmax, or applies the rejection
 * rule when sampling (§3.1), and the KV cache is rolled back by length
 * (Appendix A.1).
 *
 * Conventions for every entry point
 *   - All pointers are DEVICE pointers unless the comment says "host".  The
 *     caller allocates every buffer (workspace, weights, inputs, outputs)
 *     and keeps it alive while work that uses it is in flight.  The library
 *     never allocates device memory and never synchronises the stream
 *     (except ws_load_weights, which finishes its copies before returning).
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL
 *     is the legacy default stream).  Launch sequences are CUDA-graph
 *     capturable once the context exists.
 *   - Return value: WS_OK (0) or a negative WS_E* code.  Argument errors are
 *     detected on the host before anything is enqueued; ws_last_error()
 *     gives a one-line description.  No call aborts or throws.
 *   - Device-side invariant violations (a position at or beyond max_pos, a
 *     token id outside the vocabulary) skip the offending access and set a
 *     device status word; ws_status() reads and clears it.
 *   - "Request slots" are integers in [0, max_batch); a call works on the
 *     slots listed in `req_ids` (device int32[n_req]), in that order.
 *     Distinct entries are required.
 *   - Row-major layouts; "[n, H]" means n rows of H elements.
 *   - Model dtype: WS_F32 (float) or WS_BF16 (bfloat16, fp32 accumulation,
 *     fp32 residual stream and logits).
 */
#ifndef WS_H_
#define WS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ws_ctx ws_ctx;   /* opaque; owns no PyTorch objects */
typedef void* ws_stream;        /* cudaStream_t */

enum {
  WS_OK = 0,
  WS_EINVAL = -1,        /* bad argument (null pointer, size, mode) */
  WS_ENOSPACE = -2,      /* workspace smaller than ws_query_workspace() */
  WS_EPOS = -3,          /* a block would pass the decoder context max_pos */
  WS_ECUDA = -4,         /* a CUDA runtime / driver call failed */
  WS_EDEVICE = -5,       /* device status word was set (see ws_status) */
  WS_EUNSUPPORTED = -6   /* shape or option the library does not implement */
};

enum { WS_F32 = 0, WS_BF16 = 1 };

/* GEMM engine: both compute every output element with a K order that does
 * not depend on the number of rows, so block verification and one-token
 * decoding give bit-identical rows.  A context uses one engine throughout. */
enum { WS_GEMM_AUTO = 0, WS_GEMM_SIMT = 1, WS_GEMM_TC = 2 };

/* Model description.  Shapes of Whisper large-v3: 32 / 1280 / 20 / 5120 /
 * 51866 / 448 (Whisper-Flash §1, Appendix A.2). */
typedef struct {
  int32_t n_layers;        /* target decoder layers */
  int32_t d_model;         /* width d; multiple of 128 */
  int32_t n_heads;         /* d_model / n_heads must be 64 */
  int32_t d_ff;            /* FFN width; multiple of 128 */
  int32_t vocab;           /* V (even, at most 65,536) */
  int32_t max_pos;         /* decoder context (learned positions), <= 448 */
  int32_t drafter_layers;  /* 0 (no drafter) or 2 */
  int32_t n_hist;          /* history layers (1..8) */
  int32_t hist_layers[8];  /* zero-based target layers whose residual streams feed the drafter */
  int32_t K;               /* mask positions per draft block, <= 15 */
  int32_t dtype;           /* WS_F32 or WS_BF16 */
  int32_t max_batch;       /* request slots */
  int32_t max_frames;      /* encoder frames per request, <= 1500 */
  int32_t max_block;       /* largest verify block height H (>= K+1, >= prompt length), <= 16 */
  int32_t eos_id;          /* end-of-transcript token id */
  int32_t gemm;            /* WS_GEMM_* */
} ws_model_desc;

/* Bytes of device workspace the context needs (weights copy, caches,
 * activations, scratch).  0 if the description is invalid. */
size_t ws_query_workspace(const ws_model_desc* desc);

/* Create a context inside `workspace` (device, >= ws_query_workspace bytes,
 * 256-byte aligned) and copy the weight blobs into it.  Blobs may be host or
 * device memory, in the model dtype, laid out as:
 *   target : tok_emb[V,d] pos_emb[max_pos,d] layer*n_layers lnf_g[d] lnf_b[d]
 *   drafter: fuse_w[d, n_hist*d] lnh_g[d] lnh_b[d] mask_emb[d] lnf_g[d] lnf_b[d]
 *            layer*drafter_layers            (NULL when drafter_layers == 0)
 *   layer  : w_qkv[3d,d] w_o[d,d] w_qc[d,d] w_kvc[2d,d] w_oc[d,d]
 *            w_fc1[f,d] w_fc2[d,f] b_q b_v b_o b_qc b_vc b_oc [d]
 *            b_fc1[f] b_fc2[d] ln1_g ln1_b ln2_g ln2_b ln3_g ln3_b [d]
 * Matrices are [out, in] (y = x W^T + b); keys have no bias (Whisper).
 * The context state lives in the workspace; the host-side handle is freed
 * by ws_free.  Synchronises `stream` before returning. */
int ws_load_weights(ws_ctx** out, const ws_model_desc* desc, void* workspace,
                    size_t workspace_bytes, const void* target_blob,
                    const void* drafter_blob, ws_stream stream);

/* Reset request slots: target cache length L = 0, drafter history empty. */
int ws_reset(ws_ctx* ctx, int n_req, const int32_t* req_ids, ws_stream stream);

/* Per-request acoustic K/V (Whisper-Flash Appendix A.5: every request
 * refreshes the acoustic key/value projections of target and drafter; they
 * are written once and only read afterwards).  For every target layer and
 * every drafter layer: K_c = A W_k^T, V_c = A W_v^T + b_v.
 *   enc          [sum_i F_i, d] model dtype, requests packed back to back
 *   cu_frames    [n_req+1] int32 prefix sums of F_i (cu_frames[0] = 0)
 *   valid_frames [n_req] int32 frames that attention may see (<= F_i), or
 *                NULL (= F_i).  Frames at or beyond it are excluded from the
 *                softmax (padding), not zero-filled.
 *   max_frames_call  host int, max_i F_i (sizes the launch; <= max_frames)
 *   total_frames     host int, sum_i F_i = rows of `enc` (bounds every read
 *                    of `enc`; must equal cu_frames[n_req]) */
int ws_cross_kv(ws_ctx* ctx, int n_req, const int32_t* req_ids, const void* enc,
                const int32_t* cu_frames, const int32_t* valid_frames,
                int max_frames_call, int total_frames, ws_stream stream);

/* Block verification (Whisper-Flash §3.1): one causal target pass over
 * block[i, 0:block_len[i]] at positions L..L+block_len-1 of each request.
 * Row j attends to cache positions 0..L+j.  The block's K/V are written into
 * the paged cache (they become valid only when ws_accept advances L), and
 * the residual streams after the history layers are kept for the drafter.
 *   H          host int, row stride of block/target/logits (1..max_block)
 *   block      [n_req, H] int32 token ids (column 0 = the anchor)
 *   block_len  [n_req] int32 in 0..H (0 = request idle this call)
 *   target     [n_req, H] int32 out: greedy argmax of each row (Eq. 1,
 *              ties to the lowest id); -1 for rows >= block_len
 *   logits     [n_req, H, V] float out, or NULL (needed for sampling)
 * Prefill is a verify of the prompt with L = 0 (Appendix A.1). */
int ws_verify(ws_ctx* ctx, int n_req, const int32_t* req_ids, int H,
              const int32_t* block, const int32_t* block_len, int32_t* target,
              float* logits, ws_stream stream);

/* Parallel drafting (Whisper-Flash §3.2, Eq. 2, Appendix A.2).  First folds
 * the rows left by the last ws_verify into the drafter history (fusion
 * projection of the n_hist residual streams, LN, per-layer K/V with RoPE at
 * their absolute positions), then runs the drafter on
 * X_t = [Emb(anchor), m, ..., m] at RoPE positions t..t+K, t = L.
 *   block      [n_req, K+1] int32 in/out: column 0 (anchor) is read,
 *              columns 1..K receive the proposals
 *   temperature  0 = greedy proposals (argmax); > 0 = each mask row sampled
 *              independently from softmax(z/T) (Appendix A.4) with Philox
 *              counter (slot, round, j, 0)
 *   q_logits   [n_req, K, V] float out (draft logits), or NULL (greedy) */
int ws_draft(ws_ctx* ctx, int n_req, const int32_t* req_ids, int32_t* block,
             float temperature, uint64_t seed, uint64_t round, float* q_logits,
             ws_stream stream);

enum { WS_ACCEPT_GREEDY = 0, WS_ACCEPT_SAMPLE = 1, WS_ACCEPT_FORCED = 2, WS_ACCEPT_TREE = 3 };

/* Inputs and outputs of ws_accept (all device int32 unless noted). */
typedef struct {
  int32_t mode;              /* WS_ACCEPT_* */
  int32_t H;                 /* row stride of block / target / p_logits (TREE: the tree's rows) */
  const int32_t* block;      /* [n, H] the verified block */
  const int32_t* block_len;  /* [n] 1 + proposals; 0 = idle */
  const int32_t* target;     /* [n, H] target argmax per row (GREEDY, FORCED, TREE) */
  const float* p_logits;     /* [n, H, V] target logits (SAMPLE) */
  const float* q_logits;     /* [n, K, V] draft logits (SAMPLE) */
  float temperature;         /* SAMPLE */
  uint64_t seed, round;      /* Philox key and round (SAMPLE) */
  int32_t* budget;           /* [n] in/out output tokens left R */
  int32_t* done;             /* [n] in/out; done requests are skipped */
  int32_t* n_acc;            /* [n] out accepted candidates a */
  int32_t* n_emit;           /* [n] out tokens emitted this call */
  int32_t* next_block;       /* [n, Hn] out: column 0 = next anchor */
  int32_t next_stride;       /* Hn (>= 1) */
  int32_t* next_len;         /* [n] out: 1 + min(K, R-1) for the next block, 0 when done */
  int32_t* transcript;       /* [n, tcap] emitted tokens appended, or NULL */
  int32_t* out_len;          /* [n] in/out transcript length (required with transcript) */
  int32_t tcap;
  int32_t* n_done;           /* [1] +1 per request that finishes here, or NULL */
} ws_accept_args;

/* Acceptance and rollback (Whisper-Flash §3.1, Appendix A.1, A.4).
 * GREEDY: a = longest prefix of candidates equal to the target's argmax at
 *   the previous row; emit them plus the target's token at the first
 *   disagreement (or the bonus after all agree); an accepted EOS ends the
 *   transcript with no bonus.
 * SAMPLE: candidate j accepted iff u_j * q_j(y_j) < p_j(y_j) (FP32), u_j
 *   from Philox (slot, round, j, 1); at the first rejection a token is drawn
 *   from the normalised (p_j - q_j)_+ (or p_j when that is empty), after a
 *   full accept the bonus is drawn from row n_prop — counter (slot, round,
 *   j, 2), inverse CDF in ascending id order.  Same temperature and token
 *   suppression as the drafter.
 * FORCED: all block tokens are given (prompt prefill); emits the argmax of
 *   the last row.
 * TREE: the block is the candidate tree of ws_set_tree, verified by
 *   ws_verify_tree (Alignment Drift App. E.3).  From the root, step to the
 *   lowest-numbered child row whose token equals the target's argmax at the
 *   current row, at most R - 1 times; emit the path's tokens plus the
 *   target's token at its last row (none after an accepted EOS).  The
 *   path's self keys/values (every target layer), history rows and readout
 *   queries then move from their tree rows to block rows 1..a, so the cache
 *   holds the accepted tokens at positions L+1..L+a as after a linear
 *   acceptance.
 * Then L <- L + 1 + a (the old anchor plus the accepted candidates), R -= n_emit,
 * done when EOS was emitted or R == 0. */
int ws_accept(ws_ctx* ctx, int n_req, const int32_t* req_ids,
              const ws_accept_args* args, ws_stream stream);

/* Synthetic proposals from a reference trajectory (a workload generator,
 * not part of the method): for the anchor at t = L, candidate j (1..K) is
 * ctok[i, t, j-1] when cmask[i, t, j-1] != 0, else traj[i, t+j].
 *   block  [n, K+1] in/out (columns 1..K written)
 *   traj   [n, tlen] int32 (prompt + transcript, absolute positions)
 *   cmask  [n, max_pos, K] uint8; ctok [n, max_pos, K] int32 */
int ws_draft_synthetic(ws_ctx* ctx, int n_req, const int32_t* req_ids, int32_t* block,
                       const int32_t* traj, int tlen, const uint8_t* cmask,
                       const int32_t* ctok, ws_stream stream);

/* Truncated verification and confidence-threshold stopping (Whisper-Flash
 * Table A5 verifies only the first K' of the K proposals; Alignment Drift
 * Table 21 stops drafting when confidence falls below a threshold).  Between
 * ws_draft and ws_verify: decides how many drafted proposals each request
 * sends to verification and copies the block into the verify layout.
 *   block      [n, stride_in] int32, the drafted block (column 0 anchor,
 *              columns 1..K proposals); stride_in >= K + 1
 *   q_logits   [n, K, V] float draft logits written by ws_draft, or NULL
 *              when threshold <= 0
 *   k_verify   0..K proposals at most (K' of Table A5)
 *   threshold  proposals stop before the first position j whose confidence
 *              q_j(y_j) -- the drafter's FP32 softmax probability of its
 *              own token at `temperature` (1 when temperature is 0) -- is
 *              below it; <= 0: no threshold
 *   block_out  [n, stride_out] int32 out: columns 0..k_verify of block
 *              (stride_out >= k_verify + 1: pass stride_out as ws_verify's H)
 *   block_len  [n] int32 in/out: in, 1 + the proposals the budget allows
 *              (ws_accept's next_len; 0 = request finished); out,
 *              1 + the proposals kept (0 stays 0)
 * The output equals autoregressive greedy output for every k_verify and
 * threshold (only fewer candidates are checked). */
int ws_draft_limit(ws_ctx* ctx, int n_req, const int32_t* req_ids, const int32_t* block, int stride_in,
                   const float* q_logits, int k_verify, float threshold, float temperature,
                   int32_t* block_out, int stride_out, int32_t* block_len, ws_stream stream);

/* Candidate trees (Alignment Drift App. E.3: the drafter's ranked tokens
 * fill a fixed tree, the target verifies every node in one pass under a
 * tree attention mask, and the longest root path that matches the
 * target's argmax is accepted; a one-branch tree is the linear block).
 *   n_nodes  rows of the tree, the root (the anchor) included, 1..max_block
 *            (at most 16); 0 removes the tree
 *   parent   [n_nodes] host int32: parent[0] = -1, 0 <= parent[j] < j
 *   rank     [n_nodes] host int32: row j at depth k takes the rank[j]-th most
 *            likely token of the drafter's mask row k (0 = its argmax;
 *            equal logits rank the lower id first), 0..15; rank[0] = 0
 * Depths must not exceed K when the context has a drafter.  Host-only; the
 * tree is read when ws_tree_tokens / ws_verify_tree / ws_accept(TREE) are
 * called (a captured graph keeps the tree it was captured with). */
int ws_set_tree(ws_ctx* ctx, int n_nodes, const int32_t* parent, const int32_t* rank);

/* Fill the tree's tokens from the drafter's logits.
 *   block      [n, stride_in] int32 (device): column 0 = the anchor
 *   q_logits   [n, K, V] float (device): ws_draft's logits (suppressed ids
 *              are already -inf there)
 *   block_out  [n, stride_out] int32 out, stride_out >= n_nodes: column 0
 *              the anchor, column j the token of tree row j
 *   block_len  [n] int32 in/out: in 0 = request finished (stays 0); out
 *              min(n_nodes, max_pos - L), the tree's first rows that fit
 *              the cache (a prefix of rows is a tree) */
int ws_tree_tokens(ws_ctx* ctx, int n_req, const int32_t* req_ids, const int32_t* block, int stride_in,
                   const float* q_logits, int32_t* block_out, int stride_out, int32_t* block_len,
                   ws_stream stream);

/* Tree verification: ws_verify with H = n_nodes of the tree, where row j is
 * embedded at position L + depth(j) and attends to the cache positions
 * before L and to its ancestors' rows (itself included); row j's keys and
 * values go to cache slot L + j until ws_accept(TREE) commits the path.
 * Arguments as for ws_verify. */
int ws_verify_tree(ws_ctx* ctx, int n_req, const int32_t* req_ids, int H,
                   const int32_t* block, const int32_t* block_len, int32_t* target,
                   float* logits, ws_stream stream);

/* Verification-attention readout and windowed drafter cross-attention
 * (Alignment Drift §5 and App. D.2: the target's audio attention at one
 * decoder layer, averaged over heads, is read from the existing acoustic
 * keys after each verify; its peak frame centres a fixed-width window on
 * the drafter's cross-attention, App. A.2, +-400 ms = +-20 frames).
 *   layer       target layer whose cross-attention is read (0..n_layers-1),
 *               or -1 to switch the readout off
 *   half_width  > 0: every ws_draft restricts the drafter's cross-attention
 *               of each request to frames max(0, c - half_width) <= f <
 *               min(F, c + half_width + 1), c the request's current centre
 *               (every frame until its first readout); 0: unrestricted
 * With a readout layer set, ws_verify keeps that layer's cross-attention
 * queries of its block rows (the kernel-per-operation path is used).
 * Host-only; no device work.  Acceptance is unchanged, so greedy output
 * stays equal to autoregressive greedy output. */
int ws_set_readout(ws_ctx* ctx, int layer, int half_width);

/* The readout after ws_accept: for each request, softmax over its valid
 * frames of q k_f / sqrt(64) per head at the readout layer, averaged over
 * heads (in head order, fp32), for block row row[i] of the last ws_verify
 * (the row whose output became the next anchor: ws_accept's n_acc); its
 * peak frame (lowest on ties) becomes the request's window centre.
 *   row  [n] int32 (device) */
int ws_readout(ws_ctx* ctx, int n_req, const int32_t* req_ids, const int32_t* row, ws_stream stream);

/* Copy the current window centres of the listed slots into out [n] int32
 * (-1: none yet). */
int ws_get_centers(ws_ctx* ctx, int n_req, const int32_t* req_ids, int32_t* out, ws_stream stream);

/* Sample rows of given logits with the drafter's sampler: out[i, r] ~
 * softmax(logits[i, r, :] / T) using Philox counter (slot, round, r+1, 0).
 *   logits [n, rows, V] float; out [n, rows] int32 (row stride `rows`). */
int ws_sample(ws_ctx* ctx, int n_req, const int32_t* req_ids, const float* logits,
              int rows, float temperature, uint64_t seed, uint64_t round,
              int32_t* out, ws_stream stream);

/* Token suppression shared by draft and target logits (Appendix A.4):
 * mask [ceil(V/32)] uint32 device bitmask (bit set = id suppressed), or NULL
 * to clear.  The pointer is kept; the buffer must outlive the context. */
int ws_set_suppress(ws_ctx* ctx, const uint32_t* mask);

/* Copy the target cache lengths L of the listed slots into out [n] int32. */
int ws_get_lengths(ws_ctx* ctx, int n_req, const int32_t* req_ids, int32_t* out,
                   ws_stream stream);

/* Synchronise `stream`, return and clear the device status word (0 = ok). */
int ws_status(ws_ctx* ctx, ws_stream stream, int32_t* host_status);

/* Name of the GEMM engine in use ("simt" or "tcgen05"). */
const char* ws_gemm_engine(const ws_ctx* ctx);

/* Dataflow block verification (Whisper-Flash §3.1: the target scores the
 * anchor and the proposals in one decoder pass).  A context with one request
 * slot (max_batch 1), bf16, the tcgen05 engine, d_model a multiple of 256 up
 * to 1280, d_ff a multiple of d_model and max_pos <= 576 runs every
 * ws_verify call as one cooperative kernel (one CTA per SM): the work of
 * each step is cut into tasks that wait only on counters of the tasks whose
 * outputs they read, and each SM streams its weight tiles ahead through
 * shared memory independently of those waits.  Its rows agree with the
 * kernel-per-operation path within the bf16 tolerance, not bit for bit, and
 * a context should keep one setting for a whole decode (both settings give
 * speculative output bit-identical to autoregressive output).  Off by
 * default.
 *   enable  1: use it when eligible; 0: never (the default); -1: query only.
 * Returns 1 when eligible calls take the dataflow path, 0 when not, or
 * WS_EINVAL for a null context.  Host-only; no device work. */
int ws_fused_verify(ws_ctx* ctx, int enable);

/* Layer norm inside the projection GEMMs (Whisper-Flash §3.1 block
 * verification runs the target's pre-LN decoder layers: a LayerNorm before
 * self-attention, cross-attention and the MLP).  A bf16 context on the tcgen05 engine normalises the
 * residual rows inside the split-K GEMM that consumes them when a call has
 * at most 16 rows, instead of running a separate layer-norm kernel; the
 * normalised operand is bit-identical either way.  On by default.
 *   enable  1: use it when eligible (the default); 0: never; -1: query only.
 * Returns 1 when on, 0 when off, or WS_EINVAL for a null context.
 * Host-only; no device work. */
int ws_fused_layernorm(ws_ctx* ctx, int enable);

/* CUDA-graph replay of a fixed call sequence (Whisper-Flash Appendix A.5
 * replays prefill, drafting and each verification length from captured
 * graphs).  Between ws_capture_begin and ws_capture_end every ws_* call on
 * `stream` is recorded instead of executed (none of them synchronises);
 * ws_capture_end instantiates the graph.  Pointers and host scalars are
 * frozen at capture; device-resident state (cache lengths, blocks, budgets)
 * is read at replay.  ws_graph_launch enqueues one replay on `stream`. */
typedef struct ws_graph ws_graph;
int ws_capture_begin(ws_ctx* ctx, ws_stream stream);
int ws_capture_end(ws_ctx* ctx, ws_stream stream, ws_graph** out);
int ws_graph_launch(ws_graph* graph, ws_stream stream);
void ws_graph_free(ws_graph* graph);

/* Greedy choice over given logits rows without allocating anything.
 * The paper has no counterpart: this is an interface convenience.  Callers
 * that cannot call cudaMalloc — code running during CUDA-graph capture
 * (allocation is not capturable), code inside a host framework whose own
 * pool owns all device memory, latency-critical threads that must not block
 * on the driver — get argmax_v logits[r, v] (lowest id on ties, suppressed
 * ids skipped) for each row, the same values ws_verify returns as `target`
 * for the logits it writes.
 *   logits  [rows, vocab] float (device); out [rows] int32 (device)
 *   suppress  optional [ceil(vocab/32)] uint32 bitmask (device), or NULL
 * Scratch is a fixed 256 KB array inside the library (held by every GPU
 * that loads it until the process exits); rows > 1024 return WS_EINVAL.
 * The array's device address belongs to one CUDA context: the first call in
 * each context (the primary context of a device, a context the caller
 * created and made current, a new primary context after cudaDeviceReset)
 * looks it up with that context current and caches it for that context
 * only, so that first call should come before any stream capture.  Calls
 * share the array: calls whose work overlaps on the GPU (other streams,
 * other unordered threads) race.  A CUDA error already pending on the
 * calling thread is returned as WS_ECUDA without launching anything.
 * Errors: ws_last_error(NULL). */
int ws_argmax_rows_noalloc(const float* logits, int rows, int vocab, const uint32_t* suppress,
                           int32_t* out, ws_stream stream);

/* Number of CUDA kernels this library has launched in the process so far
 * (all contexts; host-side counter, for instrumentation). */
unsigned long long ws_launch_count(void);

/* Last error message for ctx (or for the calling thread when ctx is NULL). */
const char* ws_last_error(const ws_ctx* ctx);

/* Destroy the host handle (the workspace stays owned by the caller). */
void ws_free(ws_ctx* ctx);

/* ------------------------------------------------------------------------
 * Audio encoder (the step before the decoding path: Whisper-Flash App. B.2,
 * Table A2, once speculation removes most decoder calls the encoder takes
 * 15-34% of request time at batch one and about half at batch 32-96).  The
 * pages do not print its layers; this is the published Whisper audio
 * encoder: conv1 (n_mels -> d, kernel 3, padding 1) + GELU, conv2 (d -> d,
 * kernel 3, stride 2, padding 1) + GELU, + sinusoidal positions
 * P[t, i] = sin(t w_i), P[t, d/2 + i] = cos(t w_i), w_i = 10000^(-i/(d/2-1)),
 * n_layers pre-LN blocks (non-causal attention over the window's frames,
 * GELU MLP), and a final layer norm.  bf16 weights and activations, fp32
 * accumulation and residual stream; needs the tcgen05 engine.  Same
 * conventions as the decoder context (caller-owned workspace, asynchronous
 * calls, negative WS_E* codes, no aborts).
 * ------------------------------------------------------------------------ */
typedef struct ws_enc ws_enc;

typedef struct {
  int32_t n_layers, d_model, n_heads, d_ff;   /* large-v3: 32, 1280, 20, 5120; n_layers 1..128, d_model a
                                                 multiple of 128 up to 2048 with 64 per head, d_ff a
                                                 multiple of 128 */
  int32_t n_mels;                             /* 128 (large-v3), 80 (tiny); 1..1024 */
  int32_t n_frames;                           /* output positions F (1500 for 30 s); input 2F mel frames; <= 16384 */
  int32_t max_batch;                          /* windows per ws_encode call; 1..256 */
} ws_encoder_desc;

/* Workspace bytes for the encoder (weights, repacked convolutions, position
 * table, activations for max_batch windows); 0 if the description is invalid. */
size_t ws_encoder_workspace(const ws_encoder_desc* desc);

/* Create an encoder inside `workspace` (device, 256-byte aligned) and copy
 * the bf16 weight blob (host or device) into it:
 *   conv1_w[d, n_mels, 3] conv1_b[d] conv2_w[d, d, 3] conv2_b[d]
 *   layer * n_layers: ln1_g[d] ln1_b[d] w_qkv[3d, d] b_q[d] b_v[d] w_o[d, d]
 *                     b_o[d] ln2_g[d] ln2_b[d] w_fc1[f, d] b_fc1[f] w_fc2[d, f] b_fc2[d]
 *   lnp_g[d] lnp_b[d]
 * Convolution weights are [out, in, tap]; matrices [out, in]; no key bias.
 * Synchronises `stream` before returning. */
int ws_encoder_load(ws_enc** out, const ws_encoder_desc* desc, void* workspace, size_t workspace_bytes,
                    const void* blob, ws_stream stream);

/* Encode n windows (0 <= n <= max_batch).
 *   mel  [n, n_mels, 2F] bf16 (device): log-mel features, time innermost
 *   out  [n, F, d] bf16 (device): the encoder states A, ready for
 *        ws_cross_kv as n packed requests of F frames each
 * Device-side timeouts of bounded waits set the status word (ws_encoder_status). */
int ws_encode(ws_enc* enc, int n, const void* mel, void* out, ws_stream stream);

/* Attention kernel of the encoder: 1 = tcgen05 flash attention (S and O in
 * tensor memory, the default), 0 = the legacy mma.sync kernel (kept for
 * comparison), -1 = query only.  Returns the mode in use, or WS_EINVAL for a
 * null encoder.  Host-only. */
int ws_encoder_attention(ws_enc* enc, int mode);

/* Synchronise `stream`, return and clear the encoder's device status word. */
int ws_encoder_status(ws_enc* enc, ws_stream stream, int32_t* host_status);

/* Last error message of enc (or of the calling thread when enc is NULL). */
const char* ws_encoder_error(const ws_enc* enc);

/* Destroy the encoder's host handle (the workspace stays owned by the caller). */
void ws_encoder_free(ws_enc* enc);

#ifdef __cplusplus
}
#endif
#endif /* WS_H_ */
