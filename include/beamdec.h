/*
 * libbeamdec — the wide-beam decode step of generative recommendation, as a
 * C ABI over hand-written CUDA kernels for sm_103a (GB300).
 *
 * One decode step of request r (beam_width W, top_k K, decode step t):
 *
 *   beam_select       log-softmax of every live beam's logits over the whole
 *                     vocabulary, the catalog-trie mask of valid next codes,
 *                     per-beam top_k, global top-W over the W x top_k pool,
 *                     cumulative scores, parents, child nodes and the next
 *                     slot-table rows.
 *                     ("Generative recommendation design", xLLM, §4.1.1 beam
 *                     expansion, §4.3 early filtering, §6 beam search then
 *                     cache select; FlashRec: fused SID trie, CSR.)
 *   beam_attn_decode  split-KV beam attention: the shared stage over the
 *                     prompt KV (stored once, read once for all beams), the
 *                     unshared stage over each beam's decode-token KV reached
 *                     through the slot table, and the online-softmax merge.
 *                     ("Generative recommendation design" §4.2.1, §4.2.2.)
 *   beam_trie_build   catalog of semantic ids -> canonical CSR trie.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller, unless its
 *   comment says host.  Tensors are dense, row-major, in the layout given.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Compute entry points only enqueue work: they never synchronise the host,
 *   never allocate, and return as soon as the kernels are launched.
 * - Overlap between calls: beam_select's kernels let a kernel launched after
 *   them with programmatic stream serialization begin while they drain; such
 *   a kernel must execute griddepcontrol.wait before it reads any output of
 *   the selection.  beam_attn_decode launches its kernels that way: they read
 *   q and the prompt K/V (and, with E4M3 KV, nothing else) before waiting,
 *   and slot_table, n_live and the unshared K/V only after the previous
 *   kernel in the stream has completed.  A kernel the caller launches just
 *   before beam_attn_decode that itself lets dependents begin early must have
 *   finished writing q and the prompt K/V by then; kernels that do not (the
 *   default) give the usual stream order.
 * - Return value: BEAMDEC_OK or a negative BEAMDEC_ERR_* code.  Argument
 *   errors are detected on the host before anything is launched.  Errors a
 *   kernel detects (a slot index out of range, a bounded wait that ran out)
 *   are recorded in the status word at the start of the workspace and read
 *   with beamdec_read_status.  Kernels never trap or print.
 * - Workspace: caller-owned device memory of at least the size returned by
 *   the matching *_workspace_size query, 256-byte aligned, zero-filled
 *   before its first use (its first 256 bytes hold the status word and
 *   counters that must start at zero; the library keeps them consistent
 *   afterwards).  A workspace may be reused across calls on one stream;
 *   calls that run concurrently need separate workspaces.
 * - Bounded waits: every device-side wait (grid barrier, mbarrier) gives up
 *   after a fixed number of polls and records BEAMDEC_ERR_TIMEOUT.  Three
 *   uint32 words of a workspace are test hooks of those waits, zero in normal
 *   use (the library never writes them): bytes 12-15 replace the grid
 *   barrier's default poll count when nonzero; bytes 16-19 (beam_select
 *   workspaces) add that many arrivals to the grid barrier of the
 *   large-pool selection, which no block ever supplies, so its waits run
 *   out; bytes 20-23 (beam_attn_decode and beam_lmhead_lse workspaces), when
 *   nonzero, make each CTA of the tensor-core kernels first wait that many
 *   polls on an mbarrier that nothing completes, before it issues any copy
 *   or MMA, so the wait runs out and the CTA exits with the timeout status.
 *   Tests use them to reach the timeout path without faulting or hanging a
 *   GPU.
 */
#ifndef BEAMDEC_H
#define BEAMDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define BEAMDEC_OK 0
#define BEAMDEC_ERR_INVALID_ARG (-1)   /* NULL pointer, bad size, bad enum    */
#define BEAMDEC_ERR_UNSUPPORTED (-2)   /* legal but outside supported limits  */
#define BEAMDEC_ERR_WORKSPACE (-3)     /* workspace smaller than required     */
#define BEAMDEC_ERR_CUDA (-4)          /* a CUDA runtime call failed          */
#define BEAMDEC_ERR_TIMEOUT (-5)       /* a bounded device wait ran out       */
#define BEAMDEC_ERR_DEVICE_CHECK (-6)  /* a kernel found an index out of range */
#define BEAMDEC_ERR_ALLOC (-7)         /* beam_trie_build could not allocate  */

/* ---- element types ----------------------------------------------------- */
#define BEAMDEC_F32 0    /* IEEE binary32                                   */
#define BEAMDEC_BF16 1   /* bfloat16                                         */
#define BEAMDEC_E4M3 2   /* OCP fp8 E4M3FN, with a per-kv-head float scale   */
/* kv_dtype of beam_attn_decode only: E4M3 KV whose prompt part the
 * workspace already holds as bf16 (beam_attn_prepare_prompt). */
#define BEAMDEC_E4M3_PREPARED 3

/* ---- limits ------------------------------------------------------------ */
#define BEAMDEC_MAX_BEAM_WIDTH 8192     /* W: beam index fits 13 bits        */
#define BEAMDEC_MAX_VOCAB 262144        /* V: token fits 18 bits             */
#define BEAMDEC_MAX_LEVELS 8            /* trie levels                        */
#define BEAMDEC_MAX_CODES 65536         /* codes per level                    */

/* Human-readable name of a status code (static string). */
const char* beamdec_error_string(int status);

/* Library version as "major.minor.patch" (static string). */
const char* beamdec_version(void);

/*
 * Reads the device status word a kernel may have set in `workspace` (the
 * first 4 bytes of a beam_select or beam_attn_decode workspace), writes it to
 * *host_status (BEAMDEC_OK when clean) and clears it.  Synchronises `stream`.
 */
int beamdec_read_status(void* workspace, void* stream, int32_t* host_status);

/*
 * The step before the selection, with the selection's normaliser fused in:
 * logits = hidden x weight^T over the whole vocabulary (bf16 in, fp32
 * accumulate), reduced inside the GEMM to each row's log-sum-exp, while only
 * the token columns [window_start, window_start + window_len) - the current
 * SID level's code range - are written out.  "Generative recommendation
 * design" (xLLM) §4.3 filters invalid items before they become candidates:
 * the full [rows, V] logits never reach HBM, and beam_select then runs with
 * lse_in = lse_out on the window (it reads only the trie children's logits
 * when lse_in is given).
 *   hidden      [rows][hidden_dim] bf16, row-major, 16-byte aligned
 *   weight      [V][hidden_dim] bf16 (the LM head, one row per token)
 *   hidden_dim  multiple of 64
 *   lse_out     [rows] fp32, ln sum_v exp(logit[row, v])
 *   logits_out  fp32 rows of logits_row_stride floats; only the window's
 *               columns are written (pass stride >= V and the same pointer to
 *               beam_select).  May be NULL when window_len is 0.
 * The workspace (beam_lmhead_workspace_size bytes, 256-byte aligned) holds
 * per-tile partials; it needs no clearing.
 * Errors: INVALID_ARG, UNSUPPORTED (hidden_dim not a multiple of 64, V above
 * BEAMDEC_MAX_VOCAB), WORKSPACE, CUDA.
 */
int beam_lmhead_workspace_size(int rows, int V, size_t* bytes);
int beam_lmhead_lse(const void* hidden, const void* weight, int rows, int hidden_dim, int V,
                    int window_start, int window_len, float* lse_out, float* logits_out,
                    int64_t logits_row_stride, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Per-kernel timing for benchmarks.  beamdec_profile_enable(1) clears the
 * record and brackets every following kernel launch with a CUDA event pair
 * on its stream (at most 8192 launches are kept); beamdec_profile_enable(0)
 * stops recording.  beamdec_profile_read synchronises the recorded events and
 * returns the total milliseconds and launch count of one kernel id:
 * 0 bd_expand_kernel (selection when lse_in is given), 1 bd_global_kernel,
 * 2 bd_attn_shared_simt_kernel, 3 bd_attn_shared_tc_kernel, 4 bd_attn_merge_kernel,
 * 5 bd_kv_e4m3_to_bf16_kernel, 6 bd_stream_select_kernel (the whole selection
 * step otherwise), 7 bd_lmhead_kernel, 8 bd_lmhead_lse_kernel, 9 bd_seed_kernel
 * (open-vocabulary selection).  Host-side state is process-wide; use from one host thread.
 */
int beamdec_profile_enable(int on);
/* The same with a choice of kernels: bit k of kernel_mask brackets kernel id
 * k (ids above); 0 stops recording like beamdec_profile_enable(0).  Fewer
 * event pairs disturb the timed launches less. */
int beamdec_profile_enable_mask(unsigned kernel_mask);
int beamdec_profile_read(int kernel_id, float* total_ms, int* launches);
const char* beamdec_kernel_name(int kernel_id);

/* ======================================================================== *
 * Catalog trie
 * ======================================================================== */

/*
 * Opaque handle to a trie resident in device memory.
 *
 * Canonical form ("Generative recommendation design" §4.3 early filtering;
 * FlashRec's fused SID trie in CSR form): items are de-duplicated; the nodes
 * of level t are the distinct length-t prefixes numbered in lexicographic
 * order (level 0 holds only the root, node 0); a node's children are its
 * distinct next codes in ascending order; the child reached through edge e of
 * level t is node e of level t+1 (edges enumerate the length-(t+1) prefixes
 * in lexicographic order).  At the last level, edge e is item e of the
 * de-duplicated, lexicographically sorted catalog.
 */
typedef struct beamdec_trie beamdec_trie;

/*
 * Builds the trie of a catalog.
 *   items_host       HOST [n_items][levels] int32 codes, item-major.
 *   n_items          >= 1.
 *   levels           1..BEAMDEC_MAX_LEVELS.
 *   codes_per_level  HOST [levels]; codes of level l lie in [0, C_l),
 *                    1 <= C_l <= BEAMDEC_MAX_CODES.
 *   token_base       HOST [levels]; the vocabulary id of code c at level l is
 *                    token_base[l] + c ("Deploying FlashRec": each SID level
 *                    is a contiguous token range); token_base[l] + C_l <= vocab.
 *   vocab            vocabulary size V, <= BEAMDEC_MAX_VOCAB.
 *   stream           stream for the uploads.
 *   out              receives the handle; free it with beam_trie_free.
 * Allocates device memory (the only entry point that does).  Synchronises
 * `stream` before returning.  Errors: INVALID_ARG (a code outside [0, C_l),
 * bad sizes), UNSUPPORTED, ALLOC, CUDA.
 */
int beam_trie_build(const int32_t* items_host, int64_t n_items, int levels,
                    const int32_t* codes_per_level, const int32_t* token_base,
                    int32_t vocab, void* stream, beamdec_trie** out);

/* Frees the handle and its device memory (NULL is a no-op). */
void beam_trie_free(beamdec_trie* trie);

/*
 * Shape of the trie: levels, vocab, number of distinct items, and per level
 * (arrays of length >= levels, any may be NULL) the node count, the edge count
 * and the largest child count of any node.
 */
int beam_trie_info(const beamdec_trie* trie, int* levels, int32_t* vocab,
                   int64_t* n_distinct_items, int64_t* n_nodes, int64_t* n_edges,
                   int32_t* max_children);

/*
 * Device pointers of one level's CSR arrays, owned by the handle:
 *   off   [n_nodes + 1] int32 edge offsets (children of node n are edges
 *         off[n] .. off[n+1]-1);
 *   code  [n_edges] int32 codes, ascending within each node.
 */
int beam_trie_export(const beamdec_trie* trie, int level, const int32_t** off,
                     const int32_t** code);

/*
 * Dense child masks for one level (the FlashRec announcement's fused SID trie
 * has a dense and a CSR form).  Bit c of node n's mask (ceil(C/32) 32-bit words
 * per node, device memory owned by the trie) is set when code c is one of n's
 * children.  While a level has masks, beam_select, beam_select_gumbel and
 * beam_select_fixed_lse enumerate that level's candidates from the mask (bit
 * order = code order = child order) instead of the CSR code list; without
 * lse_in that takes two launches (the rows' normalisers are streamed first,
 * then the rows expanded) instead of one.  The selections are identical
 * either way.  beam_trie_make_dense
 * builds them from the level's CSR (a host round trip on `stream`,
 * synchronised); beam_trie_drop_dense frees them; beam_trie_export_dense
 * returns the device pointer (NULL without masks) and words per node.
 * Errors: INVALID_ARG (bad level), UNSUPPORTED (C > 16384, or masks above
 * 1 GiB), ALLOC, CUDA.
 */
int beam_trie_make_dense(beamdec_trie* trie, int level, void* stream);
int beam_trie_drop_dense(beamdec_trie* trie, int level);
int beam_trie_export_dense(const beamdec_trie* trie, int level, const uint32_t** mask, int32_t* words);

/* ======================================================================== *
 * Beam selection
 * ======================================================================== */

/*
 * Workspace bytes for beam_select with R requests, beam width W, top_k K and
 * vocab V (pool W x min(K, V) keys per request plus counters).
 */
int beam_select_workspace_size(int R, int W, int K, int V, size_t* bytes);

/*
 * One expansion step for R requests ("Generative recommendation design"
 * §4.1.1: every beam expands top_k candidates, beam_width beams are kept from
 * the beam_width x top_k pool; §4.3: invalid paths never become candidates;
 * §6: cache selection after the reorder).
 *
 * Inputs (device):
 *   logits      fp32; the row of beam b of request r starts at
 *               logits + (r*W + b) * row_stride and holds V values.
 *               Only rows b < n_live_in[r] are read.  Values must be finite.
 *   row_stride  elements between consecutive beam rows (>= V).
 *   lse_in      optional [R][W] fp32: when not NULL, the log-sum-exp of each
 *               live row is taken from here instead of being computed (e.g.
 *               when the producer of the logits already has it).
 *   cum_in      [R][W] fp32 cumulative log-probability of each live beam.
 *   node_in     [R][W] int32 trie node of each live beam at level `level`
 *               (ignored when trie is NULL).
 *   n_live_in   [R] int32 live beams per request, 0..W (beams 0..n-1 live).
 *   slot_in     [R][W][T] int32 slot rows of the live beams; entries
 *               0..step-1 are read.
 *   trie        catalog trie, or NULL for open-vocabulary decoding (every
 *               token is a candidate).
 *   level       trie level the beams sit at (0 <= level < trie levels).
 *   step        decode step t (0 <= step < T); the token chosen by output
 *               beam j at this step is assigned slot step*W + j.
 *   R, W, K, V, T  requests, beam width (<= 8192), top_k (>= 1), vocab
 *               (<= 262144, must equal the trie's vocab), slots per beam row.
 * Outputs (device, [R][W] unless noted), rank-ordered by
 * (score desc, parent asc, token asc):
 *   tokens      int32 chosen token, -1 for rows j >= n_live_out[r].
 *   parents     int32 index of the parent beam in the input, -1 if dead.
 *   cum_out     fp32 score s = fl32(cum_in[parent] + fl32(logit - lse)),
 *               round-to-nearest-even, no FMA; -inf if dead.
 *   lse_out     optional fp32 log-sum-exp of each live input row (NULL to skip);
 *               entries of rows b >= n_live_in[r] are left untouched.
 *   node_out    int32 child node at level+1 (= edge index); at the last level
 *               the item index; -1 for open vocabulary or dead rows.
 *   n_live_out  [R] int32 = min(W, pool size).
 *   slot_out    [R][W][T] int32: entries 0..step-1 copied from the parent's
 *               row, entry step = step*W + j, later entries -1; dead rows -1.
 * No output may overlap an input (the kernels write outputs while other
 * blocks still read inputs); slot_out == slot_in, cum_out == cum_in,
 * node_out == node_in and n_live_out == n_live_in are rejected.
 * Per beam, candidates are ranked by (score desc, token asc) and the first
 * min(top_k, #candidates) enter the pool.
 * Errors: INVALID_ARG, UNSUPPORTED (W, V, K limits; a trie node with more
 * children than the supported maximum), WORKSPACE, CUDA.
 */
int beam_select(const float* logits, int64_t row_stride, const float* lse_in,
                const float* cum_in, const int32_t* node_in, const int32_t* n_live_in,
                const int32_t* slot_in, const beamdec_trie* trie, int level, int step,
                int R, int W, int K, int V, int T,
                int32_t* tokens, int32_t* parents, float* cum_out, float* lse_out,
                int32_t* node_out, int32_t* n_live_out, int32_t* slot_out,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * beam_select with temperature > 0: Gumbel top-k.  "Deploying FlashRec"
 * (serving parameters): a positive temperature makes the selection Gumbel
 * top-k, the noise only orders the candidates and the returned sequence score
 * does not include it.  Here each candidate (request r, step t, beam b, token
 * v) with score s = fl32(cum + fl32(logit - lse)) is ordered (per beam, then
 * per request, ties as in beam_select) by the key
 *     fl32(fl32(s * fl32(1 / temperature)) + g),
 *     g = -ln(-ln(u)),  u = ((word0 >> 9) + 1/2) * 2^-23,
 * word0 = first output word of Philox4x32-10 (Salmon et al., SC 2011) at
 * counter (v, b, r, t) and key (seed & 0xffffffff, seed >> 32); ln is a
 * float32 atanh-series logarithm with every step rounded to nearest.  The
 * same seed, step and inputs give the same selection.  cum_out holds s (no
 * noise); every other argument, output and error is as for beam_select, and
 * the workspace is the same size.
 * Errors: INVALID_ARG also for temperature <= 0, not finite, or so small that
 * 1 / temperature overflows float32.
 */
int beam_select_gumbel(const float* logits, int64_t row_stride, const float* lse_in,
                       const float* cum_in, const int32_t* node_in, const int32_t* n_live_in,
                       const int32_t* slot_in, const beamdec_trie* trie, int level, int step,
                       int R, int W, int K, int V, int T, float temperature, uint64_t seed,
                       int32_t* tokens, int32_t* parents, float* cum_out, float* lse_out,
                       int32_t* node_out, int32_t* n_live_out, int32_t* slot_out,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * beam_select_fixed_lse - the one-launch selection (the kernel beam_select
 * runs when lse_in is NULL: every live row streamed for its log-sum-exp,
 * then expanded and selected in the same launch) with the candidates scored
 * against a caller-supplied normaliser.  "Generative recommendation design"
 * §4.1.1 (the beam_width x top_k pool and the global top beam_width): the
 * selection is a function of the float32 candidate scores, so a reference
 * implementation that rounds its own normaliser can check this kernel's
 * decisions bit for bit only when both sides score against the same float32
 * value.
 *   score_lse  [R][W] fp32 (device, required): candidate scores are
 *              s = fl32(cum_in[b] + fl32(logit - score_lse[b])); read for
 *              live rows only.
 *   lse_out    still receives the kernel's OWN log-sum-exp of every live row
 *              (NULL to skip), computed exactly as in beam_select.
 *   temperature, seed  0 for deterministic top-k, or a positive temperature
 *              for Gumbel top-k exactly as in beam_select_gumbel.
 * Every other argument, output, limit and error is as for beam_select
 * (lse_in does not exist here), and the workspace is the same size.
 * Errors: INVALID_ARG also for a NULL score_lse or a temperature that is
 * neither 0 nor valid for beam_select_gumbel.
 */
int beam_select_fixed_lse(const float* logits, int64_t row_stride, const float* score_lse,
                          const float* cum_in, const int32_t* node_in, const int32_t* n_live_in,
                          const int32_t* slot_in, const beamdec_trie* trie, int level, int step,
                          int R, int W, int K, int V, int T, float temperature, uint64_t seed,
                          int32_t* tokens, int32_t* parents, float* cum_out, float* lse_out,
                          int32_t* node_out, int32_t* n_live_out, int32_t* slot_out,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * beam_select_static — beam_select without a caller-provided workspace.
 * The pages have no counterpart to this entry point; it serves callers of
 * this library that cannot allocate device memory: a plugin interface that
 * hands the library only its input and output buffers, or a process whose
 * device memory belongs to another allocator, so that cudaMalloc may not be
 * called on the calling path.
 *
 * Arguments, outputs, ordering and errors are those of beam_select, minus
 * `workspace` / `workspace_bytes`.  The scratch is one file-scope device
 * array of BEAMDEC_STATIC_SELECT_BYTES bytes, which every GPU that loads the
 * library holds until the process exits; shapes whose
 * beam_select_workspace_size exceeds it are rejected with
 * BEAMDEC_ERR_UNSUPPORTED before anything is launched.  Nothing is allocated.
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it with the current context (a call under a
 * different context looks it up again): make that first call before any
 * stream capture.  Resetting the device (cudaDeviceReset) while the library
 * stays loaded is not supported.  Arguments are checked before the array is
 * touched, so a refused call writes nothing.  All calls on a device share the array and it keeps the last
 * call's contents; each call clears the status word and counters it needs on
 * its own stream first, so calls in stream order are independent, but calls
 * that overlap on the GPU (unordered streams) race on the array.  The status
 * word in the array is cleared at the start of each call and is not readable
 * through beamdec_read_status; use beam_select with an own workspace to
 * observe device-side checks.
 */
#define BEAMDEC_STATIC_SELECT_BYTES ((size_t)16 << 20)
int beam_select_static(const float* logits, int64_t row_stride, const float* lse_in,
                       const float* cum_in, const int32_t* node_in, const int32_t* n_live_in,
                       const int32_t* slot_in, const beamdec_trie* trie, int level, int step,
                       int R, int W, int K, int V, int T,
                       int32_t* tokens, int32_t* parents, float* cum_out, float* lse_out,
                       int32_t* node_out, int32_t* n_live_out, int32_t* slot_out, void* stream);

/* ======================================================================== *
 * Beam attention
 * ======================================================================== */

/*
 * Workspace bytes for beam_attn_decode (partial (max, sum, output) triples of
 * the shared stage, one per prompt split and query row; sized for the split
 * path even when the merge runs inside the shared stage).
 */
int beam_attn_workspace_size(int R, int W, int Hq, int Hkv, int d, int max_prompt_len,
                             int kv_dtype, size_t* bytes);

/*
 * Split-KV attention for one decode step ("Generative recommendation design"
 * §4.2.1: shared KV = the prompt's prefill KV stored once for all beams,
 * unshared KV = one entry per decode token per beam; §4.2.2: shared stage,
 * unshared stage, OnlineSoftmax merge).
 *
 * For request r, live beam j < n_live[r] and query head h (kv head
 * g = h / (Hq/Hkv)):
 *   out[r][j][h] = softmax(sm_scale * q . k_i) v_i over the prompt rows of r
 *                  followed by the unshared slots slot_table[r][j][0..step];
 * rows j >= n_live[r] are written as zeros.
 *
 *   q               [R][W][Hq][d]  q_dtype (F32 or BF16).
 *   shared_k/v      [sum P][Hkv][d] kv_dtype; request r owns rows
 *                   prompt_offsets[r] .. prompt_offsets[r+1]-1.
 *   prompt_offsets  [R+1] int32, non-decreasing, prompt_offsets[0] = 0.
 *   max_prompt_len  host int >= every P_r (sizes the launch).
 *   shared_rows     host copy of prompt_offsets[R]: the rows of shared_k /
 *                   shared_v (<= R * max_prompt_len).  No row at or beyond it
 *                   is read; a device-side mismatch with prompt_offsets[R]
 *                   sets BEAMDEC_ERR_DEVICE_CHECK.
 *   unshared_k/v    [R][T*W][Hkv][d] kv_dtype: the per-request slot pool.
 *   slot_table      [R][W][T] int32; entries 0..step of live rows must lie in
 *                   [0, T*W) (checked in-kernel; a bad slot sets
 *                   BEAMDEC_ERR_DEVICE_CHECK in the status word and is skipped).
 *   n_live          [R] int32.
 *   k_scale/v_scale [Hkv] fp32 dequantisation scales, required for E4M3 KV,
 *                   ignored otherwise (may be NULL).
 *   sm_scale        softmax scale (pass 0 for 1/sqrt(d)).
 *   out             [R][W][Hq][d] out_dtype (F32 or BF16).
 * Supported: d in {64, 128}; Hq % Hkv == 0; Hq/Hkv <= 16; q/kv/out dtypes
 * F32/F32/F32, BF16/BF16/BF16, BF16/E4M3/BF16 (and BF16/E4M3_PREPARED/BF16
 * after beam_attn_prepare_prompt on the same workspace).  BF16 queries with d = 128
 * and a group size dividing 128 take the tensor-core shared stage (fp8 KV is
 * first dequantised to bf16 in the workspace); other shapes run it on CUDA
 * cores.  When that stage covers every prompt in one split (at most 6
 * unshared tokens, q / unshared K, V / out 16-byte aligned, BF16 output),
 * the unshared stage and the merge run in its epilogue and the partials
 * never leave the kernel; otherwise a merge kernel reads them from the
 * workspace.  The tensor-core stage (and the fp8 dequantisation) launch as
 * programmatic dependents of the previous kernel in the stream (see the
 * conventions above).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 */
int beam_attn_decode(const void* q, const void* shared_k, const void* shared_v,
                     const int32_t* prompt_offsets, int max_prompt_len, int64_t shared_rows,
                     const void* unshared_k, const void* unshared_v,
                     const int32_t* slot_table, const int32_t* n_live, int step,
                     int R, int W, int Hq, int Hkv, int d, int T,
                     int q_dtype, int kv_dtype, int out_dtype,
                     const float* k_scale, const float* v_scale, float sm_scale,
                     void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The prompt part of E4M3 KV, dequantised once into an attention workspace
 * (the prompt KV of a request is fixed for all of its decode steps, while
 * beam_attn_decode with BEAMDEC_E4M3 rewrites this bf16 copy on every call).
 * Later beam_attn_decode calls on the same workspace pass kv_dtype
 * BEAMDEC_E4M3_PREPARED with the same shared_k, shared_v and shared_rows:
 * they read the copy and skip the dequantisation, so the shared stage can
 * also start while the previous kernel drains (see the conventions above).
 * The copy is exact (every e4m3 value is a bf16 value; the per-head scales
 * are applied later, as without it).  The workspace records the two
 * pointers and shared_rows; a PREPARED call with others sets
 * BEAMDEC_ERR_DEVICE_CHECK in its status word.  A caller that rewrites the
 * prompt KV in place must prepare again.
 *
 *   shared_k/v, prompt_offsets, max_prompt_len, shared_rows, R, W, Hq, Hkv, d:
 *       as for beam_attn_decode (W and Hq size the workspace's layout).
 *   kv_dtype  BEAMDEC_E4M3 (other types have nothing to prepare: the call
 *             returns BEAMDEC_OK without launching anything; so do shapes
 *             the tensor-core stage does not take, which read fp8 directly).
 *   workspace as for beam_attn_decode (sized with BEAMDEC_E4M3).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 */
int beam_attn_prepare_prompt(const void* shared_k, const void* shared_v, const int32_t* prompt_offsets,
                             int max_prompt_len, int64_t shared_rows, int R, int W, int Hq, int Hkv, int d,
                             int kv_dtype, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BEAMDEC_H */
