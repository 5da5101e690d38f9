/*
 * bi.h -- C ABI of libbi: batch-invariant reduction kernels for GB300 (sm_103a).
 *
 * The three reductions of an LLM forward pass -- RMSNorm, the linear-layer
 * GEMM and attention over a paged KV cache -- written so that every output
 * row is a function of its own inputs only: the same bytes whatever the batch
 * size, the row's position in the batch, the neighbouring rows, the KV-cache
 * length of other requests or the way a prompt is cut into prefill chunks.
 *
 * Pages this interface follows:
 *   [P1] "Reproducible LLM Inference - Batch Invariance, the Cost of
 *        Determinism, and Where Bitwise Identity Is Actually Required"
 *        (hidekazu-konishi.com)
 *   [P3] "Your Answer Depends on Who Else Is in the Batch" (praveentn.live)
 * Batch invariance is defined in P1 §5.1: the result for one element of a
 * batch does not change when the batch changes.  P1 §5.3-5.5 name the three
 * operations and the freedom each kernel must give up.
 *
 * Conventions (all entry points):
 *   - Tensor pointers are DEVICE pointers owned by the caller; bf16 means IEEE
 *     bfloat16 (passed as void*), row-major, densely packed unless a stride is
 *     given.  Every tensor pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous on that stream; they never synchronise
 *     and never allocate device memory.  Scratch space ("workspace") is
 *     provided by the caller; its size comes from the matching *_workspace_size
 *     query, which is pure host arithmetic except where noted.
 *   - Return: BI_OK, or an error code; on an argument error nothing is
 *     launched.  Errors found on the device (a page id outside the pool, a
 *     kv length beyond the page table, a bounded wait that ran out) do not
 *     fault the GPU: the kernel skips the access, records the code in a
 *     per-device error word and returns; bi_check_device_errors reads it.
 *   - Modes: BI_MODE_INVARIANT is the batch-invariant kernel.  BI_MODE_VARIANT
 *     is the same arithmetic with the reduction split chosen from the batch
 *     shape (split-K for the GEMM, a split row for RMSNorm, a fixed split
 *     COUNT for attention), i.e. what a shape-tuned kernel does; it is
 *     deterministic run to run but not batch-invariant, and exists to measure
 *     the cost of invariance (P1 §8).
 *   - Only the current CUDA device is used.
 */
#ifndef BI_H
#define BI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bi_status {
  BI_OK = 0,
  BI_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned pointer */
  BI_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement */
  BI_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
  BI_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  BI_ERR_DEVICE_BOUNDS = 5, /* device-side check: index outside a buffer */
  BI_ERR_TIMEOUT = 6        /* device-side bounded wait ran out */
} bi_status;

typedef enum bi_mode {
  BI_MODE_INVARIANT = 0,
  BI_MODE_VARIANT = 1
} bi_mode;

/* ------------------------------------------------------------------------ */
/* RMSNorm  (P1 §5.3-5.4; P3 "Where the reductions are", "A Concrete Example") */
/* ------------------------------------------------------------------------ */
/* y[i,:] = x[i,:] * (mean_j x[i,j]^2 + eps)^(-1/2) * w
 *   x [M,H] bf16, w [H] bf16, y [M,H] bf16 (y may not alias x).
 *   y_f32 (may be NULL): [M,H] fp32, the same values before the final
 *   rounding to bf16.
 *   Sum of squares in fp32; one rounding to bf16 at the end.
 * INVARIANT: one row per thread block; the block shape and the order of the
 *   in-row reduction depend on H only (P1 §5.3: more rows only means more
 *   rows per core).  Needs no workspace.
 * VARIANT: when M is small the row is cut into s chunks reduced by separate
 *   blocks and combined in a second pass (P1 §5.3; P3's 32-block example);
 *   s is chosen from M and the SM count.  Workspace: see below.
 * Requirements: H % 8 == 0, 8 <= H <= 65536, M >= 0 (M == 0 is a no-op).
 * Errors: BI_ERR_INVALID_ARG (null/misaligned), BI_ERR_UNSUPPORTED (H),
 *   BI_ERR_WORKSPACE, BI_ERR_CUDA. */
bi_status bi_rmsnorm(const void* x, const void* w, void* y, float* y_f32, int64_t M,
                     int64_t H, float eps, bi_mode mode, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Residual add fused with RMSNorm (the pre-norm step of a decoder layer).
 * The pages define only RMSNorm ("Your Answer Depends on Who Else Is in the
 * Batch", "A Concrete Example"); the fused add is this library's addition:
 *   h = bf16(x + residual)   (each element: fp32 add, rounded once to bf16),
 *       written over residual (the updated residual stream);
 *   y = RMSNorm(h) * w        exactly as bi_rmsnorm(h, w, y, ...).
 * The bytes equal a bf16 add followed by bi_rmsnorm, in both modes; the
 * invariant mode reads x and residual once (one row per CTA, the RMSNorm
 * row reduction above).  Layouts, alignment and errors as bi_rmsnorm; x and
 * residual must not overlap.  BI_MODE_VARIANT runs the add, then the split
 * RMSNorm, and needs bi_rmsnorm_workspace_size(M, H, BI_MODE_VARIANT)
 * bytes. */
bi_status bi_add_rmsnorm(const void* x, void* residual, const void* w, void* y, float* y_f32,
                         int64_t M, int64_t H, float eps, bi_mode mode, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Bytes of workspace bi_rmsnorm needs: 0 for BI_MODE_INVARIANT; for
 * BI_MODE_VARIANT an upper bound (M * 64 * 4).  Host arithmetic only. */
size_t bi_rmsnorm_workspace_size(int64_t M, int64_t H, bi_mode mode);

/* ------------------------------------------------------------------------ */
/* GEMM  (P1 §3.3, §5.4; P3 "Where the reductions are")                     */
/* ------------------------------------------------------------------------ */
/* C[i,n] = sum_k A[i,k] * W[n,k]
 *   A [M,K] bf16 (activations, K contiguous), W [N,K] bf16 (a Linear weight,
 *   K contiguous), C [M,N] bf16.  fp32 accumulation in tensor memory, one
 *   rounding to bf16 at the end.
 * INVARIANT: one tensor-core instruction family (tcgen05.mma kind::f16,
 *   M=128, K=16) and one K order (k-blocks of 64 in increasing k) for every
 *   M; no split-K, no stream-K (P1 §5.4: the instruction and the split are
 *   the two freedoms to give up).  Output tiles are 128 x 64 (instruction
 *   N=64) for M <= 64 when ceil(N/64) tiles fit in one wave of the device's
 *   SMs, K % 64 == 0 and K >= 256 (more blocks then stream the weight);
 *   otherwise 128 x 192 above 32 rows when its tiles fill the SMs' rounds
 *   better (rounds of #SM tiles times the width, 192's weighted by 10/9),
 *   else 128 x 256.  The instruction's N does not change any output
 *   element's sum (every element has the same bytes at N = 64, 192 and 256
 *   on sm_103a), so a row's bytes do not depend on M.  Needs no
 *   workspace.
 * VARIANT: same tiles and instruction, but K is split into s slices chosen
 *   from M, N and the SM count (split-K, P1 §5.4: only when the output tiles
 *   cover at most a quarter of the SMs, then doubling until the slices cover
 *   them, at least 4 k-blocks per slice); fp32 slice results are
 *   summed in slice order by a second kernel.  s = variant_splits if > 0.
 * Requirements: M >= 0, N >= 1, K >= 1, N % 8 == 0, K % 8 == 0 (16-byte rows
 *   for the tensor-memory-access engine), all dims < 2^31.
 * Errors: as bi_rmsnorm. */
bi_status bi_gemm(const void* A, const void* W, void* C, int64_t M, int64_t N, int64_t K,
                  bi_mode mode, int variant_splits, void* workspace,
                  size_t workspace_bytes, void* stream);

/* Bytes of workspace bi_gemm needs: 0 for BI_MODE_INVARIANT.  For
 * BI_MODE_VARIANT it queries the current device's SM count (so it needs a
 * GPU) and returns splits * M * N * 4 for the split count bi_gemm will use;
 * (size_t)-1 if the device cannot be queried. */
size_t bi_gemm_workspace_size(int64_t M, int64_t N, int64_t K, bi_mode mode,
                              int variant_splits);

/* Split count bi_gemm uses in BI_MODE_VARIANT for this shape on a device
 * with num_sms SMs (1 = no split), counted over the tiles bi_gemm runs for
 * it (above); bi_gemm_swiglu uses the count of its [M, 2F] shape.  Host
 * arithmetic only. */
int bi_gemm_variant_splits(int64_t M, int64_t N, int64_t K, int num_sms);

/* Gate/up projection with the SwiGLU product in the GEMM epilogue (P1 §5.4:
 * element-wise work is batch-invariant by nature, so fusing it into the
 * invariant GEMM keeps every row's bytes).
 *   out[i,j] = bf16( silu(g) * u ),  silu(x) = x / (1 + exp(-x)) in fp32,
 *   g = bf16((A W^T)[i, 256*(j/128) + j%128]),
 *   u = bf16((A W^T)[i, 256*(j/128) + 128 + j%128]).
 *   A [M,K] bf16, W [2F,K] bf16 with the gate and up rows stacked in blocks
 *   of 128 features (rows 256b .. 256b+127: gate of features 128b ..
 *   128b+127; rows 256b+128 .. 256b+255: up of the same features), out [M,F]
 *   bf16.  The GEMM arithmetic (instruction, K order, split count in both
 *   modes) is bi_gemm's on (M, 2F, K), always with 128 x 256 tiles (a tile
 *   holds the gate and up rows of 128 features), so out holds exactly the
 *   bytes of bi_gemm into a [M,2F] buffer followed by bi_silu_mul with
 *   block = 128, with no [M,2F] tensor written.
 * Workspace: bi_gemm_workspace_size(M, 2F, K, mode, variant_splits) bytes.
 * Requirements: F % 128 == 0, K % 8 == 0, 2F and K < 2^31; pointers 16-byte
 *   aligned.  Errors: as bi_gemm. */
bi_status bi_gemm_swiglu(const void* A, const void* W, void* out, int64_t M, int64_t F,
                         int64_t K, bi_mode mode, int variant_splits, void* workspace,
                         size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Attention over a paged KV cache  (P1 §5.5; P3 "The attention detail that */
/* gets missed")                                                            */
/* ------------------------------------------------------------------------ */
/* Common layout:
 *   k_cache, v_cache [num_pages][Hkv][page_size][D] bf16.  Token t of
 *     sequence b lives in page block_table[b*max_blocks_per_seq + t/page_size]
 *     at slot t % page_size.  The caller writes the K/V of new tokens into
 *     the cache and extends block_table / kv_lens BEFORE calling attention,
 *     so cached and new tokens are read from one layout and reduced alike
 *     (P1 §5.5).
 *   block_table [B][max_blocks_per_seq] int32, kv_lens [B] int32: device.
 *   Grouped-query attention: q-head h reads kv-head h / (Hq/Hkv).
 *   scores = sm_scale * q.k (pass 1/sqrt(D) for the usual scale; sm_scale
 *   must be positive and finite, else BI_ERR_INVALID_ARG); softmax over the
 *   visible keys; out = sum softmax * v.
 *   out is bf16; out_f32 (may be NULL) receives the same values before the
 *   final rounding, in fp32, same layout.
 * Split plan (BI_MODE_INVARIANT, P1 §5.5 fixed split SIZE): the keys
 *   0..L-1 of a query are cut at multiples of split_size; each chunk is
 *   reduced with an online softmax over key tiles of 64 in increasing order
 *   (partial max m, sum l, unnormalised o), and the chunks are merged by a
 *   left fold in chunk order with the log-sum-exp rule, then o times the
 *   correctly rounded 1/l is rounded.
 *   Boundaries depend on absolute key indices only, never on L, B, the grid
 *   or the chunking of a prompt.
 * BI_MODE_VARIANT (a split plan sized from the batch, the kind of plan the
 *   pages name as not batch-invariant): one chunk size C for the call,
 *   C = 64 * max(ceil(Hkv * T / U), ceil(T_max / c)), where T is the sum and
 *   T_max the largest of the sequences' 64-key tile counts ceil(L/64),
 *   U = 4 * (resident split-kernel blocks on the device) the target number
 *   of work units, and c = variant_splits if > 0, else
 *   c = min(128, ceil(max_kv_len / 256)) the largest number of chunks a
 *   sequence may get (it sizes the workspace);
 *   sequence b is cut at multiples of C into ceil(L_b / C) chunks.  Every
 *   boundary moves with the lengths of the other sequences in the call.
 * A sequence with L == 0 produces zeros.
 * Requirements: D in {64, 128}; Hq % Hkv == 0 and Hq/Hkv <= 16;
 *   page_size == 16; split_size a positive multiple of 64; num_pages >= 1;
 *   max_blocks_per_seq >= 1.
 * Device checks: a page id outside [0, num_pages) or a kv length above
 *   max_blocks_per_seq*page_size (or above max_kv_len) is recorded as
 *   BI_ERR_DEVICE_BOUNDS and the offending sequence is skipped. */

/* Decode: one new query token per sequence.
 *   q [B][Hq][D] bf16, out [B][Hq][D] bf16.
 *   max_kv_len: host-side upper bound on kv_lens (sizes the grid only).
 *   Workspace: bi_attn_decode_workspace_size(...) bytes. */
bi_status bi_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, const int32_t* kv_lens, void* out,
                         float* out_f32, int B, int Hq, int Hkv, int D, int page_size,
                         int64_t num_pages, int max_blocks_per_seq, int max_kv_len,
                         int split_size, float sm_scale, bi_mode mode,
                         int variant_splits, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Bytes of workspace bi_attn_decode needs: the unit list of the split plan
 * (16 bytes per (sequence, split)) and the split partials m, l, o in fp32,
 * i.e. 256 + up256(16*B*S_max) + up256(8*B*Hq*E) + 4*B*Hq*S_max*D with
 * S_max = ceil(max_kv_len / split_size) (the variant's count in
 * BI_MODE_VARIANT), E = S_max rounded up to an even number and up256
 * rounding up to a multiple of 256.
 * Host arithmetic, except that BI_MODE_VARIANT with variant_splits <= 0
 * queries the current device's SM count ((size_t)-1 if that fails). */
size_t bi_attn_decode_workspace_size(int B, int Hq, int Hkv, int D, int max_kv_len,
                                     int split_size, bi_mode mode, int variant_splits);

/* Decode without a caller workspace, for callers that cannot allocate device
 * memory (an engine that has given all of HBM to its KV-cache pool and
 * forbids further allocations, a plugin whose host framework owns the
 * allocator).  The pages describe no such entry point; it is a convenience of
 * this library.
 * Same arguments, layout and result as bi_attn_decode in BI_MODE_INVARIANT
 * (bit-identical output), minus mode and workspace.  The scratch comes from a
 * fixed array of BI_NOALLOC_SCRATCH_BYTES inside the library, reserved on
 * every GPU that loads this code until the process exits; the call itself
 * allocates nothing.
 * Limit: bi_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, split_size,
 *   BI_MODE_INVARIANT, 0) must not exceed BI_NOALLOC_SCRATCH_BYTES, else the
 *   call returns BI_ERR_WORKSPACE and launches nothing.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture begins.
 * The looked-up address is kept for the life of the process: after a
 * cudaDeviceReset of that device it is stale, so do not call this entry
 * point again on a device that has been reset.
 * All calls share the array: calls whose kernels overlap on the GPU race with
 * each other, so order them (e.g. issue them on one stream).
 * Errors: as bi_attn_decode, plus BI_ERR_WORKSPACE for the size limit. */
#define BI_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
bi_status bi_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* kv_lens, void* out,
                                 float* out_f32, int B, int Hq, int Hkv, int D, int page_size,
                                 int64_t num_pages, int max_blocks_per_seq, int max_kv_len,
                                 int split_size, float sm_scale, void* stream);

/* Causal prefill of one chunk per sequence (P1 §5.5, §6.4: a prompt may
 * arrive in chunks; every token's reduction must not depend on the chunking).
 *   q [total_q][Hq][D] bf16: the chunk tokens of all sequences, sequence b
 *     owning rows cu_q[b] .. cu_q[b+1]-1 (cu_q [B+1] int32, device).
 *   q_start_pos [B] int32 (device): absolute position of sequence b's first
 *     chunk token; token i of the chunk sits at position q_start_pos[b]+i and
 *     attends to keys 0..q_start_pos[b]+i.  kv_lens[b] must be at least
 *     q_start_pos[b] + chunk length (the cache already holds the chunk).
 *   out [total_q][Hq][D] bf16 (+ optional out_f32).
 *   max_q_len: host bound on the chunk lengths; max_kv_len: host bound on
 *     kv_lens.  Both size the grid only.
 * In BI_MODE_INVARIANT the result at every position is bit-identical to
 * bi_attn_decode in BI_MODE_INVARIANT with L = position + 1 and the same
 * split_size.  BI_MODE_VARIANT sizes the chunks from max_kv_len and c
 * (split size = 64 * ceil(max_kv_len / (64 c))), so results move with the
 * chunking.  Needs no workspace (pass NULL, 0).
 * Errors: as bi_attn_decode; a block whose sequence has a page id outside
 *   the pool (among the pages its keys use) or a chunk past kv_lens records
 *   BI_ERR_DEVICE_BOUNDS before any copy and leaves its rows unwritten. */
bi_status bi_attn_prefill_chunk(const void* q, const int32_t* cu_q,
                                const int32_t* q_start_pos, const void* k_cache,
                                const void* v_cache, const int32_t* block_table,
                                const int32_t* kv_lens, void* out, float* out_f32, int B,
                                int Hq, int Hkv, int D, int page_size, int64_t num_pages,
                                int max_blocks_per_seq, int64_t total_q, int max_q_len,
                                int max_kv_len, int split_size, float sm_scale,
                                bi_mode mode, int variant_splits, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Write K/V rows of new tokens into the paged cache (the precondition of
 * both attention calls, P1 §5.5).  k_new, v_new [n_tokens][Hkv][D] bf16;
 * token i goes to sequence seq[i] at absolute position pos[i] (int32 device
 * arrays), i.e. page block_table[seq*max_blocks + pos/page_size], slot
 * pos % page_size.  Pure data movement, no arithmetic.  Bounds are checked
 * on the device as for attention. */
bi_status bi_kv_write(const void* k_new, const void* v_new, const int32_t* seq,
                      const int32_t* pos, int64_t n_tokens, void* k_cache, void* v_cache,
                      const int32_t* block_table, int Hkv, int D, int page_size,
                      int64_t num_pages, int max_blocks_per_seq, void* stream);

/* ------------------------------------------------------------------------ */
/* Element-wise decoder-layer steps (P1 §5.4: batch-invariant by nature)    */
/* ------------------------------------------------------------------------ */
/* Row gather: dst[i, :] = src[idx[i], :] for i < n (token embedding lookup,
 * or picking the rows that need logits).  src [rows][H] bf16, idx int32 [n]
 * (device), dst [n][H] bf16.  H % 8 == 0.  An index outside [0, rows) is
 * recorded in the device error word (BI_ERR_DEVICE_BOUNDS) and its row is
 * written as zeros.  Pure data movement. */
bi_status bi_gather_rows(const void* src, int64_t rows, int64_t H, const int32_t* idx, int64_t n,
                         void* dst, void* stream);

/* Rotary position embedding fused with the split of a QKV projection.
 *   qkv [T][(Hq + 2 Hkv) D] bf16: per token the Hq query heads, then the Hkv
 *   key heads, then the Hkv value heads, D elements each (the output of
 *   bi_gemm with the stacked q/k/v weight); pos int32 [T] (device): each
 *   token's absolute position.
 *   q [T][Hq][D], k [T][Hkv][D]: rotated; v [T][Hkv][D]: copied.
 * Rotation (the rotate-half arrangement): for pair i < D/2 of a head,
 *   angle = pos * theta^(-2i/D),
 *   y[i] = x[i] cos - x[i + D/2] sin,  y[i + D/2] = x[i + D/2] cos + x[i] sin.
 * The angle is formed in fp64 and reduced modulo 2 pi; sine, cosine and the
 * rotation are fp32, rounded once to bf16.  The pages fix no positional
 * encoding; this is the one of the Llama family.
 * Requirements: D % 16 == 0, D <= 1024, theta > 1.  Errors: as bi_rmsnorm. */
bi_status bi_rope_qkv(const void* qkv, const int32_t* pos, int64_t T, int Hq, int Hkv, int D,
                      double theta, void* q, void* k, void* v, void* stream);

/* SwiGLU product: out[t, j] = bf16(silu(g) * u), silu(g) = g / (1 + exp(-g))
 * in fp32, out [T][F] bf16, from the gate and up projections stacked in one
 * GEMM output gate_up [T][2F] bf16 in blocks of `block` features:
 *   g = gate_up[t, 2*block*(j/block) + j%block],  u = the element block
 *   columns further on.
 * block = F: all gate columns, then all up columns.  block = 128: the layout
 * bi_gemm writes with bi_gemm_swiglu's weight, so that this kernel after
 * bi_gemm gives the bytes of bi_gemm_swiglu.
 * Requirements: F % block == 0, block % 8 == 0, F < 2^31.  Errors: as bi_rmsnorm. */
bi_status bi_silu_mul(const void* gate_up, int64_t T, int64_t F, int64_t block, void* out,
                      void* stream);

/* ------------------------------------------------------------------------ */
/* Next-token selection  (P1 §9.2, §9.3)                                    */
/* ------------------------------------------------------------------------ */
/* One token per request from its row of logits, deterministic for given
 * (logits row, temperature, seed, step) whatever the batch around it.
 *   logits [B][V] bf16 (row-major, e.g. the LM-head output of bi_gemm);
 *   temperature [B] float, seed [B] and step [B] uint64, tokens [B] int32:
 *   all device pointers, caller-owned; logits aligned to 2 bytes, the
 *   others to their element size.
 * temperature[b] > 0: Gumbel-max sampling (P1 §9.3: the logits perturbed by
 *   Gumbel noise from a seeded hash), tokens[b] = argmax_v z_v / T + G_v with
 *   G_v = -log(-log(u_v)), computed in fp32 (z * (1/T), then + G).  u_v is
 *   drawn by Philox4x64-10 (Salmon et al., SC 2011) under key {seed[b], 0}
 *   at counter {v / 8, step[b], 0, 0}: 32-bit half v % 2 (low half first) of
 *   output word (v / 2) % 4, top 23 bits k, u = (k + 1/2) 2^-23.  The draw
 *   follows softmax(z / T); step is the caller's per-request counter (e.g.
 *   the position of the token being chosen), so successive tokens of one
 *   request get fresh noise.
 * temperature[b] <= 0 (or NaN): greedy, tokens[b] = argmax_v z_v (P1 §9.2).
 * Ties go to the lowest index; -0 equals +0; a NaN score counts as -inf (it
 *   is chosen only when no entry scores above -inf, lowest index first: an
 *   all-NaN or all -inf row gives token 0).
 * The argmax is a reduction under a total order, so its result does not
 *   depend on how the row is split; one launch: a cluster of 8 CTAs per row
 *   below 128 rows (one row keeps several SMs busy), one CTA per row above.
 * Requirements: 0 <= B <= 65535, 1 <= V < 2^31.  Needs no workspace.
 * Errors: BI_ERR_INVALID_ARG (null, misaligned, B < 0, V < 1),
 *   BI_ERR_UNSUPPORTED (B or V too large), BI_ERR_CUDA (launch). */
bi_status bi_sample(const void* logits, int64_t B, int64_t V, const float* temperature,
                    const uint64_t* seed, const uint64_t* step, int32_t* tokens, void* stream);

/* ------------------------------------------------------------------------ */
/* Errors and introspection                                                 */
/* ------------------------------------------------------------------------ */
/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns BI_OK, the first recorded device error, or BI_ERR_CUDA. */
bi_status bi_check_device_errors(void* stream);

/* Diagnostic of the failure path: launches one thread that waits on a
 * barrier nothing arrives on, with the bounded wait every kernel of this
 * library uses, given up after timeout_us microseconds (1 .. 2,000,000).
 * The kernel records BI_ERR_TIMEOUT in the device error word and returns;
 * the context stays usable.  Returns the launch status (BI_ERR_INVALID_ARG
 * for an out-of-range timeout); read the recorded status with
 * bi_check_device_errors. */
bi_status bi_selftest_wait_timeout(uint32_t timeout_us, void* stream);

/* Static English description of a status code (never NULL). */
const char* bi_status_string(bi_status status);

/* Library version, "major.minor.patch". */
const char* bi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BI_H */
