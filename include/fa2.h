/*
 * fa2.h -- C ABI of libfa2.so: FlashAttention-2 exact multi-head attention,
 * forward and backward, on one sm_103a (GB300) GPU.
 *
 * The operation (sources: the FlashAttention-2 write-ups
 *   "FlashAttention学习笔记(2)" (amentiraz.github.io), sections "V2 的运作流程"
 *       and "V2中的thread blocks排布";
 *   "大猿搬砖简记" (damodev.csdn.net), the V2 forward / backward walk-throughs;
 *   "flash-attention123和ring-attention" (blog.csdn.net), 优化1 - 优化4):
 *
 *   for every batch b and head h, with S = scale * Q K^T (N x N):
 *     causal: S[i][j] = -inf for j > i   (top-left alignment, key j visible to query i iff j <= i)
 *     O   = softmax_rows(S) V
 *     L_i = ln(sum_j exp(S[i][j]))       (the logsumexp; the only softmax statistic stored)
 *   backward, given dO:
 *     P = exp(S - L), dV = P^T dO, dP = dO V^T, D_i = sum_c dO[i][c] * O[i][c],
 *     dS = P o (dP - D), dQ = scale * dS K, dK = scale * dS^T Q.
 *
 * Layout of every tensor argument: contiguous row-major [B][H][N][d] of 16-bit
 * floats (dtype FA2_FP16 or FA2_BF16); lse is contiguous fp32 [B][H][N].
 * Q, K and V share the sequence length N (self-attention), except in
 * fa2_fwd_qk / fa2_bwd_qk, where K and V have their own length Nk.
 *
 * Ownership: the caller allocates and owns every buffer, including the
 * backward workspace. The library keeps only a per-device status word (a
 * static device variable) and never frees caller memory.
 *
 * Execution: every compute entry point only enqueues work on `stream` (a
 * cudaStream_t, or NULL for the legacy default stream) and returns; nothing
 * synchronises the host. Outputs are fully overwritten, never accumulated into,
 * and must not overlap any input.
 *
 * Errors: every entry point returns an fa2_status (int). Arguments are checked
 * before anything is launched; on an error nothing is launched and no output
 * is touched. A kernel never traps: a bounded wait that runs out writes
 * FA2_ERR_DEVICE_TIMEOUT into the device status word, which
 * fa2_get_device_status() reports.
 */
#ifndef FA2_H_
#define FA2_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa2_status {
  FA2_OK = 0,
  FA2_ERR_INVALID_ARG = 1,    /* null pointer, B/H/N < 1, bad dtype/causal, scale not finite or <= 0 */
  FA2_ERR_UNSUPPORTED = 2,    /* d not in {64, 128}, or a size beyond the documented limits */
  FA2_ERR_ALIGNMENT = 3,      /* a tensor pointer not 16-byte aligned (lse: 4-byte; workspace: 256-byte) */
  FA2_ERR_ARCH = 4,           /* current device is not compute capability 10.3 (sm_103) */
  FA2_ERR_CUDA = 5,           /* a CUDA runtime / driver call or kernel launch failed */
  FA2_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up on a bounded wait (see fa2_get_device_status) */
  FA2_ERR_WORKSPACE = 7,      /* backward workspace missing or smaller than fa2_bwd_workspace_size */
  FA2_ERR_OVERLAP = 8         /* an output buffer overlaps an input buffer */
} fa2_status;

typedef enum fa2_dtype { FA2_FP16 = 0, FA2_BF16 = 1 } fa2_dtype;

/* Forward pass (FlashAttention-2 forward: Q rows outer, K/V tiles inner, online
 * softmax with running max m and sum l, one division by l at the end, only
 * L = m + ln l stored; fully masked causal K/V tiles skipped).
 *   q, k, v : device, [B][H][N][d] dtype, 16-byte aligned, read only.
 *   o       : device, [B][H][N][d] dtype, 16-byte aligned, written.
 *   lse     : device, [B][H][N] fp32, 4-byte aligned, written (natural log).
 *   B, H, N : >= 1; B <= 65535, H <= 65535, B*H*N < 2^31.
 *   d       : 64 or 128.
 *   causal  : 0 or 1.
 *   scale   : finite, > 0 (usually 1/sqrt(d)).
 *   dtype   : FA2_FP16 or FA2_BF16 (q, k, v, o share it).
 *   stream  : cudaStream_t or NULL. */
int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
            int d, int causal, float scale, int dtype, void* stream);

/* K/V-split forward ("大猿搬砖简记", thread-block section: when the (row block,
 * batch, head) workers cannot fill the SMs, each worker's K/V range may be cut
 * into num_splits parts run by separate blocks, whose partial results are then
 * combined to recover the global softmax). num_splits is the part count of the
 * longest worker (n_max K/V tiles of 128 keys); a worker with n tiles (shorter
 * under the causal mask) gets min(n, ceil(n * num_splits / n_max)) balanced,
 * contiguous, non-empty parts. A worker with one part writes O and L itself;
 * the parts of the others write fp32 O / l and logsumexp into the workspace
 * and count their arrival per 128-row tile; the part that arrives last forms
 * L = ln sum_s exp(lse_s), O = sum_s exp(lse_s - L) O_s (no CTA waits on
 * another; the counters are zeroed on the stream before the launch). Blocks
 * are launched longest row block first, heads varying fastest.
 * Same result as fa2_fwd up to rounding.
 *   num_splits : 1 .. 128 (1 runs fa2_fwd and ignores the workspace).
 *   workspace  : device, >= fa2_fwd_split_workspace_size(...) bytes, 256-byte
 *                aligned, scratch owned by the caller (contents ignored on
 *                entry, undefined on exit).
 *   other arguments as in fa2_fwd. */
int fa2_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int N, int d, int causal, float scale, int dtype, int num_splits, void* workspace,
                  size_t workspace_bytes, void* stream);

/* Forward pass in the FlashAttention-1 loop order, for measuring the loop
 * order ("FlashAttention学习笔记(2)", the FlashAttention-1 forward algorithm
 * and the comparison of the two loop orders): K/V blocks outer, query blocks
 * inner, one CTA per (batch, head). At every (K/V block j, query block i) step
 * the running O_i (kept normalised), row max m_i and row sum l_i are read from
 * and written back to the workspace in HBM:
 *   m_new = max(m_i, m~), l_new = e^(m_i - m_new) l_i + e^(m~ - m_new) l~,
 *   O_i <- (l_i e^(m_i - m_new) O_i + e^(m~ - m_new) P~ V_j) / l_new,
 * with m~, P~ = exp(S - m~), l~ of the block S = scale Q_i K_j^T. The same
 * O and L as fa2_fwd up to rounding. Query and key lengths are equal.
 *   workspace : device, >= fa2_fwd_kv_outer_workspace_size(...) bytes,
 *               256-byte aligned, scratch owned by the caller (contents
 *               ignored on entry, undefined on exit).
 *   other arguments as in fa2_fwd. */
int fa2_fwd_kv_outer(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, int causal, float scale, int dtype, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Bytes of workspace fa2_fwd_kv_outer needs: B*H x N x (d + 2) fp32 (O_i, m_i,
 * l_i), each array rounded up to 256 bytes. Returns 0 for invalid sizes. */
size_t fa2_fwd_kv_outer_workspace_size(int B, int H, int N, int d);

/* One forward + backward step on HOST buffers: q, k, v, dO are read from host
 * memory and o, lse, dq, dk, dv written back to host memory, the copies
 * overlapped with the kernels. Every (batch, head) is independent
 * ("FlashAttention学习笔记(2)", V2中的thread blocks排布), so the B*H heads are
 * cut into chunks of heads_per_chunk consecutive heads and pipelined on three
 * internal streams: upload of chunk c+1, fa2_fwd + fa2_bwd of chunk c,
 * download of chunk c-1, with two device slots. The results are the bits of
 * fa2_fwd + fa2_bwd on device copies of the same tensors.
 *   q, k, v, dO       : host, [B][H][N][d] dtype, read only. Pinned
 *                       (page-locked) memory lets the copies overlap.
 *   o, dq, dk, dv     : host, [B][H][N][d] dtype, written.
 *   lse               : host, [B][H][N] fp32, written.
 *   heads_per_chunk   : >= 1, or 0 for ceil(B*H / 8).
 *   workspace         : device, >= fa2_step_host_workspace_size(...) bytes,
 *                       256-byte aligned, owned by the caller.
 *   stream            : a stream of the current device (or NULL). The chain
 *                       starts after the work queued on it and the stream
 *                       waits for the chain's end; host buffers must stay
 *                       valid until then. Calls on one device are enqueued
 *                       one at a time (a per-device lock).
 *   other arguments as in fa2_fwd. */
int fa2_step_host(const void* q, const void* k, const void* v, const void* dO, void* o, float* lse,
                  void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                  int dtype, int heads_per_chunk, void* workspace, size_t workspace_bytes,
                  void* stream);

/* Device workspace fa2_step_host needs: two slots, each of 8 [hc][N][d]
 * 16-bit tensors, one [hc][N] fp32 tensor and fa2_bwd's workspace for one
 * chunk (hc = heads per chunk as above); each array rounded up to 256 bytes.
 * Returns 0 for invalid sizes. */
size_t fa2_step_host_workspace_size(int B, int H, int N, int d, int heads_per_chunk);

/* Bytes of workspace fa2_fwd_split needs: num_splits x B*H x N x (d + 1) fp32
 * (the parts' O / l and logsumexp) plus B*H x ceil(N / 256) x 2 int32 arrival
 * counters, each of the three arrays rounded up to 256 bytes. Returns 0 for
 * invalid sizes. */
size_t fa2_fwd_split_workspace_size(int B, int H, int N, int d, int num_splits);

/* The split count of the same page: for each candidate s in 1 .. min(128,
 * num_sms, K/V tiles of the longest worker), the SM utilisation of the split
 * launch; returns the smallest s whose utilisation is at least 0.95 of the
 * best. The page does not define utilisation; here it is the fraction of the
 * SMs' time spent on K/V tiles, useful tiles / (num_sms * makespan), when the
 * launch's CTAs (row blocks of 256 queries longest first, each block's parts
 * in order, heads fastest) start in launch order on the SM that frees first,
 * each taking its K/V tiles plus 1 tile of fixed cost, plus 6 more if its row
 * block is split (partial write and merge) -- costs measured on GB300. 1 when
 * the unsplit launch already reaches 0.95. To split automatically, a caller
 * passes this count (with the device's SM count) to fa2_fwd_split; forward()
 * of the Python binding does so by default. Host only; results are cached
 * per shape. Returns 0 for invalid arguments. */
int fa2_num_splits(int B, int H, int N, int d, int causal, int num_sms);

/* Forward with different query and key lengths: q, o [B][H][Nq][d], lse
 * [B][H][Nq]; k, v [B][H][Nk][d]. The pages keep seqlen_q and seqlen_k
 * distinct ("FlashAttention学习笔记(2)", V2中的thread blocks排布) without stating
 * the causal mask for unequal lengths; here it is top-left: key j is visible
 * to query i iff j <= i, so query i sees keys 0 .. min(i, Nk - 1). Keys past
 * Nk are masked. Other arguments and limits as in fa2_fwd (for Nq and Nk). */
int fa2_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Nq, int Nk, int d, int causal, float scale, int dtype, void* stream);

/* Bytes of device workspace fa2_bwd needs: the fp32 row sums D = rowsum(dO o O)
 * and L * log2(e), each [B*H][N rounded up to 128], then 256 bytes for the
 * work counter of the main launch. Returns 0 for invalid sizes. */
size_t fa2_bwd_workspace_size(int B, int H, int N, int d);

/* Backward pass (FlashAttention-2 backward: D = rowsum(dO o O) first; then K/V
 * column blocks outer, Q tiles inner, S and P recomputed from L, dK/dV
 * accumulated on chip; dQ, which accumulates along the key direction, in fp32
 * on chip by a query-tile worker of its own -- no atomics, bit-reproducible).
 *   q, k, v, o, dO : device [B][H][N][d] dtype, 16-byte aligned (o and lse from fa2_fwd).
 *   lse            : device [B][H][N] fp32.
 *   dq, dk, dv     : device [B][H][N][d] dtype, 16-byte aligned, written.
 *   workspace      : device, >= fa2_bwd_workspace_size(B,H,N,d) bytes, 256-byte
 *                    aligned, scratch owned by the caller; contents on entry
 *                    are ignored and on exit undefined.
 *   other arguments as in fa2_fwd. */
int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
            const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
            float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace fa2_bwd_atomic needs: fa2_bwd's, then the fp32 dQ
 * accumulator [B*H][N rounded up to 128][d]. Returns 0 for invalid sizes. */
size_t fa2_bwd_atomic_workspace_size(int B, int H, int N, int d);

/* The same gradients as fa2_bwd, computed the way the pages' column workers
 * do it ("FlashAttention学习笔记(2)", Foward和backward中的thread block划分; "大猿
 * 搬砖简记", V2 backward): one CTA per 128-key column block keeps K_j, V_j in
 * shared memory and dK_j, dV_j in TMEM while the query tiles stream past, and
 * adds each dQ_i contribution (dS K, fp32) into an accumulator in global
 * memory with TMA reduce-adds; the preprocessing pass zeroes the accumulator
 * and a last pass writes dq = scale * accumulator. Five products per (key
 * block, query tile) pair, against seven for fa2_bwd, but on GB300 it runs
 * slower than fa2_bwd (the reduce-adds and the longer per-tile chain of the
 * compute warps); kept as the measured alternative. The order of the
 * reduce-adds varies from run to run, so dq is not bit-reproducible (dk and
 * dv are). Equal query and key lengths.
 *   workspace : >= fa2_bwd_atomic_workspace_size(B,H,N,d) bytes, 256-byte aligned.
 *   other arguments as in fa2_bwd. */
int fa2_bwd_atomic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                   void* stream);

/* Backward with different query and key lengths (mask as in fa2_fwd_qk): q, o,
 * dO, dq [B][H][Nq][d], lse [B][H][Nq]; k, v, dk, dv [B][H][Nk][d]. Keys that
 * no query sees (causal, Nk > Nq) get dk = dv = 0. The workspace is
 * fa2_bwd_workspace_size(B, H, Nq, d) bytes. Other arguments as in fa2_bwd. */
int fa2_bwd_qk(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dO, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
               int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
               void* stream);

/* fa2_bwd, plus: phase_events (4 cudaEvent_t created by the caller, or NULL)
 * are recorded on `stream` before the preprocessing kernel, between it and
 * the main launch (the dK/dV and dQ workers), and twice after the main launch,
 * so the caller can time the two launches. */
int fa2_bwd_timed(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                  void* const* phase_events, void* stream);

/* fa2_bwd_atomic with the same four phase events: before the preprocessing
 * kernel, between it and the column workers' launch, between that and the dq
 * conversion, and after it. */
int fa2_bwd_atomic_timed(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, int causal, float scale, int dtype, void* workspace,
                         size_t workspace_bytes, void* const* phase_events, void* stream);

/* fa2_bwd without a caller-provided workspace, for callers that must not
 * allocate device memory: code running inside a memory pool or a framework
 * allocator it does not own, or a process that fixes its device footprint at
 * start-up and may not call cudaMalloc afterwards. (The FlashAttention-2 pages
 * have no counterpart to this entry point; it is a property of this library.)
 * The backward's scratch -- the row sums D and L*log2(e), 8 bytes per query
 * row with rows padded to 128 per head, and a 256-byte work counter -- lives
 * in a 16 MiB + 256 byte array built into
 * the library, one per GPU that loads it, held until the process exits. Its
 * gradients are the bits of fa2_bwd on the same inputs.
 *   arguments  : as fa2_bwd, minus the workspace.
 *   limit      : fa2_bwd_workspace_size(B,H,N,d) <= 16 MiB + 256 (for example up to
 *                B*H = 256 heads of N = 8192); larger sizes return
 *                FA2_ERR_UNSUPPORTED and touch nothing.
 *   set-up     : the first call on a device looks up the array's device
 *                address with that device current and keeps it for the life
 *                of the process; make that first call before any stream
 *                capture. A device reset (cudaDeviceReset) reloads the
 *                library's device code at a new address, so do not use this
 *                entry point (or the library's status word) across a reset.
 *   concurrency: every call on a device shares the one array, so calls that
 *                may overlap on the GPU (different streams, or different host
 *                threads) race on it; serialise them. Nothing needs clearing
 *                between calls: each call writes every scratch entry it reads.
 *   allocation : none (no cudaMalloc, cudaFree or allocating library call). */
int fa2_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                    int causal, float scale, int dtype, void* stream);

/* Synchronises `stream`, then returns and clears the current device's status
 * word: FA2_OK, or FA2_ERR_DEVICE_TIMEOUT if any kernel since the last call
 * gave up on a bounded wait, or FA2_ERR_CUDA if the synchronisation failed. */
int fa2_get_device_status(void* stream);

/* Static, human-readable name of a status code. */
const char* fa2_status_string(int status);

/* ---- Host-only queries of the work mapping (no GPU needed) ----------------
 * Forward row blocks ("thread blocks" of "FlashAttention学习笔记(2)",
 * V2中的thread blocks排布) form the grid (num_m_block, B, H), the row block
 * varying fastest. Each owns rows_per_cta = 256 query rows (two 128-row
 * tiles). The split forward launches one CTA per (row block, part); the
 * unsplit one runs the row blocks on a persistent grid (fa2_fwd_schedule). */
int fa2_fwd_grid(int B, int H, int N, int grid_out[3], int* rows_per_cta);

/* Query rows [*row_begin, *row_end) and the number of K/V tiles of 128 keys
 * that forward row block `block_x` loads (causal: fully masked tiles are
 * skipped, "flash-attention123和ring-attention", 优化3). */
int fa2_fwd_block_work(int block_x, int N, int causal, int* row_begin, int* row_end,
                       int* kv_tiles);

/* Schedule of the unsplit forward on a device with num_sms multiprocessors:
 * *num_ctas CTAs (at most num_sms), each running a fixed list of row blocks.
 * Without a causal mask the row blocks are dealt round robin; with one, pairs
 * of row blocks q and num_m_block-1-q (a constant K/V total) are dealt round
 * robin, and the pairs left for a last partial round are the most balanced
 * ones of the last heads, run as halves. cta_of_block and pos_of_block (host
 * arrays of B*H*num_m_block ints, in fa2_fwd_grid order; either may be NULL)
 * receive each row block's CTA and its position in that CTA's list.
 * Returns FA2_ERR_INVALID_ARG for sizes < 1, causal not 0/1 or a NULL num_ctas. */
int fa2_fwd_schedule(int B, int H, int N, int causal, int num_sms, int* num_ctas, int* cta_of_block,
                     int* pos_of_block);

/* Backward dK/dV work = (num_n_block, B, H): one worker per 128-key column
 * block ("FlashAttention学习笔记(2)", Foward和backward中的thread block划分). The
 * main launch runs these workers, then the dQ workers, on a persistent grid
 * of at most one CTA per SM. */
int fa2_bwd_grid(int B, int H, int N, int d, int grid_out[3], int* keys_per_cta,
                 int* q_rows_per_tile);

/* Keys [*key_begin, *key_end) of backward column block `block_x` and the query
 * tiles [*q_tile_begin, *q_tile_end) (of q_rows_per_tile rows) it visits. */
int fa2_bwd_block_work(int block_x, int N, int d, int causal, int* key_begin, int* key_end,
                       int* q_tile_begin, int* q_tile_end);

/* ---- Diagnostics ----------------------------------------------------------
 * fa2_fwd, plus: tile_counts (device int array with one slot per forward row block,
 * grid order x fastest, or NULL) receives the number of K/V tiles loaded for
 * each row block. */
int fa2_fwd_instrumented(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, int causal, float scale, int dtype, int* tile_counts,
                         void* stream);

/* The CUDA runtime error code (cudaError_t; a driver CUresult plus 1000 for a
 * failed tensor-map encode) behind the last FA2_ERR_CUDA this thread received,
 * or 0. */
int fa2_last_cuda_error(void);

/* Arms a host-side fault for the next call of its kind in this process. Each
 * kind makes one TMA producer warp skip one load, so that a consumer's bounded
 * wait on it runs out after timeout_ms (1..5000) milliseconds instead of the
 * default 2 s; the kernel then records FA2_ERR_DEVICE_TIMEOUT, lets the copies
 * and MMAs it issued finish, frees its tensor memory and returns:
 *   1  the next fa2_fwd / fa2_fwd_qk / fa2_fwd_instrumented: the first V tile;
 *   2  the next fa2_fwd_split: the first V tile of every part;
 *   3  the next backward (fa2_bwd, fa2_bwd_atomic and their variants): the
 *      first dO tile of every K/V column worker;
 *   4  the next fa2_bwd (or fa2_bwd_qk, fa2_bwd_noalloc): the first V tile of
 *      every dQ worker;
 *   0  disarms.
 * Outputs of the faulted call are undefined. Exists to test the failure path
 * without hanging or faulting the GPU. */
int fa2_debug_arm_fault(int kind, int timeout_ms);

#ifdef __cplusplus
}
#endif

#endif /* FA2_H_ */
