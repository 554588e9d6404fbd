/*
 * cpattn.h - C ABI of the context-parallel causal attention library
 * (libcpattn.so), GB300 / sm_103a.
 *
 * What the library computes (all readings of the sources are listed with
 * the functions below):
 *
 *   [CP-handbook] "上下文并行：Ring Attention 与 Ulysses" (AI-infra
 *   handbooks, training / model / context parallelism):
 *     - section "哪些运算可以直接切": block attention with global query/key
 *       offsets returning the output and the per-row log-sum-exp;
 *     - self-test answers and section "Ring Attention：KV 沿环传一圈": the LSE
 *       merge lse = log(e^lse1 + e^lse2), o = o1 e^(lse1-lse) + o2 e^(lse2-lse),
 *       and the ring loop (KV passed to rank+1, later KV skipped);
 *     - section "之字形切分": the zigzag layout (2P chunks, rank r holds r and
 *       2P-1-r);
 *     - section "Ulysses：在序列和头之间转置": the seq<->head all-to-all.
 *
 * Conventions shared by every entry point
 *   - Tensors are row-major and token-major: q/out [S, H, D], k/v [S, Hkv, D]
 *     (D innermost), LSE [H, S] fp32 in natural log.  Under GQA query head h
 *     reads KV head h / (H / Hkv).
 *   - Every data pointer is caller-owned DEVICE memory unless stated; the
 *     library allocates no device memory and keeps no pointer after a call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  A return of CP_OK means the work was validated and
 *     enqueued.  Device-side waits are bounded: a kernel whose wait expires
 *     records a status that cp_check_device_error() reports.
 *   - Errors never abort or throw: every function returns a negative
 *     cp_status and stores a message readable with cp_last_error() (per
 *     thread).  Validation happens before anything is enqueued.
 *   - bf16 inputs require D = 128 (tensor-core path, fp32 accumulation);
 *     fp32 inputs accept D in {16, 32, 64, 128} (fp32 CUDA-core path).
 *     All data pointers must be 16-byte aligned.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* cp_stream_t; /* identical to cudaStream_t */

typedef enum {
  CP_OK = 0,
  CP_ERR_ARG = -1,     /* null pointer, negative size, bad enum, P out of range */
  CP_ERR_SHAPE = -2,   /* divisibility / unsupported D / H % Hkv etc.          */
  CP_ERR_DTYPE = -3,   /* unsupported dtype combination                        */
  CP_ERR_ALIGN = -4,   /* a pointer is not 16-byte aligned                     */
  CP_ERR_CUDA = -5,    /* a CUDA runtime/driver call failed                    */
  CP_ERR_TIMEOUT = -6, /* a device-side bounded wait expired (see below)       */
  CP_ERR_BOUNDS = -7   /* bounds-checked build: a kernel's bounds check failed  */
} cp_status;

typedef enum { CP_F32 = 0, CP_BF16 = 1 } cp_dtype;
typedef enum { CP_CONTIGUOUS = 0, CP_ZIGZAG = 1, CP_STRIPED = 2 } cp_layout;

/* Largest number of virtual ranks the ring accepts. */
#define CP_MAX_RANKS 16

/*
 * cp_attn_block - one block of causal attention with global offsets.
 *   [CP-handbook] section "哪些运算可以直接切" (the attention helper).
 *
 *   s[h,i,j] = scale * q[i,h,:] . k[j,h/(H/Hkv),:]
 *   masked (causal != 0) where k_offset + j > q_offset + i  (diagonal kept)
 *   lse[h,i] = log sum_j exp(s[h,i,j])
 *   out[i,h,:] = sum_j exp(s[h,i,j] - lse[h,i]) v[j,h/(H/Hkv),:]
 *
 *   q [Sq,H,D] in_dt; k, v [Sk,Hkv,D] in_dt; out [Sq,H,D] out_dt;
 *   lse [H,Sq] fp32.  scale <= 0 selects 1/sqrt(D).
 *   A row that sees no key (possible with offsets, or Sk = 0) gets
 *   lse = -inf and out = 0 (the identity of the merge).
 *   Sq = 0 is a no-op.  Sq, Sk, offsets < 2^31.
 */
int cp_attn_block(const void* q, const void* k, const void* v, cp_dtype in_dt,
                  int64_t Sq, int64_t Sk, int H, int Hkv, int D,
                  int64_t q_offset, int64_t k_offset, int causal, float scale,
                  void* out, cp_dtype out_dt, float* lse, cp_stream_t stream);

/*
 * cp_lse_merge - in-place merge acc <- acc (+) blk of two partial
 * attentions over the same rows.  [CP-handbook] self-test answers and
 * section "Ring Attention：KV 沿环传一圈".
 *
 *   lse = logaddexp(lse_acc, lse_blk)
 *   out_acc = out_acc * e^(lse_acc - lse) + out_blk * e^(lse_blk - lse)
 *   lse_acc = lse
 *
 *   out_* [Sq,H,D] fp32, lse_* [H,Sq] fp32.  -inf on one side gives that
 *   side weight 0; -inf on both gives lse -inf and out 0.
 *   D must be a multiple of 4 with D/4 a power of two or a multiple of 32.
 *   out_blk/lse_blk may not alias out_acc/lse_acc.
 */
int cp_lse_merge(float* out_acc, float* lse_acc,
                 const float* out_blk, const float* lse_blk,
                 int64_t Sq, int H, int D, cp_stream_t stream);

/*
 * cp_ring_workspace_size - bytes of device workspace cp_ring_forward /
 * cp_ring_step need: S*H*D*4 (an fp32 accumulator) when out_dt = CP_BF16,
 * else 0 (the fp32 out buffer is the accumulator).  Returns a negative
 * cp_status on bad arguments.
 */
int64_t cp_ring_workspace_size(int64_t S, int H, int D, cp_dtype out_dt);

/*
 * cp_ring_forward - causal attention of a whole sequence by the
 * Ring-Attention schedule of P virtual ranks on this GPU.
 *   [CP-handbook] sections "Ring Attention：KV 沿环传一圈" and "之字形切分".
 *
 *   q [S,H,D], k, v [S,Hkv,D] in NATURAL sequence order; the virtual ranks'
 *   shards are row sets of them, so no reorder copy is made.
 *   layout CP_CONTIGUOUS: P chunks of C = ceil(S/P) rows; rank r holds chunk r
 *   layout CP_ZIGZAG:     2P chunks of C = ceil(S/(2P)) rows; rank r holds
 *                         chunks r and 2P-1-r
 *     When the chunk count does not divide S the last chunks are shorter (or
 *     empty): the same result as padding the sequence at its end and
 *     discarding the padded rows ([CP-practice] section 7.1), without
 *     computing them.
 *   layout CP_STRIPED:    rank r holds tokens r, r+P, r+2P, ... (Striped
 *                         Attention, [SP-CP-survey] section 3.3; S % P = 0)
 *   Step t (0 <= t < P): rank r holds the KV of rank src = (r - t) mod P
 *   (received from rank r-1); it evaluates every (own query chunk, held KV
 *   chunk) pair in which some key precedes some query (for striped: every
 *   pair), merges the result into its running (out, lse) with the LSE merge,
 *   and skips the rest.
 *   Execution: with bf16 inputs (any layout) all P steps run inside one
 *   kernel launch (cp_ring_forward_fused; the workspace is then unused);
 *   with fp32 inputs one launch per step covers all ranks and merges into
 *   the accumulator (cp_ring_forward_steps).
 *   out [S,H,D] out_dt, lse [H,S] fp32.  workspace: device memory of
 *   cp_ring_workspace_size() bytes (NULL allowed when that is 0).
 *   The result equals cp_attn_block over the whole sequence up to rounding.
 *   1 <= P <= CP_MAX_RANKS.
 */
int cp_ring_forward(const void* q, const void* k, const void* v, cp_dtype in_dt,
                    int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                    void* out, cp_dtype out_dt, float* lse, void* workspace,
                    cp_stream_t stream);

/*
 * cp_ring_forward_steps - the ring of cp_ring_forward as P kernel launches,
 * one per step (every layout and dtype).  Launch t evaluates the blocks of
 * step t for all virtual ranks and LSE-merges each into the fp32
 * accumulator (the workspace, or out itself when out_dt = CP_F32) in its
 * epilogue; the last step to touch a row writes it to out.  Launches after
 * the first start while the previous one drains (programmatic dependent
 * launch) and wait for it only before their epilogue.  Arguments as
 * cp_ring_forward; same result up to rounding (bit for bit the result of
 * cp_ring_step for t = 0 .. P-1).
 */
int cp_ring_forward_steps(const void* q, const void* k, const void* v, cp_dtype in_dt,
                          int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                          void* out, cp_dtype out_dt, float* lse, void* workspace,
                          cp_stream_t stream);

/*
 * cp_ring_forward_fused - the ring of cp_ring_forward with all P steps
 * inside one kernel launch.  [CP-handbook] sections "Ring Attention：KV 沿环
 * 传一圈" and "之字形切分"; the running (max, sum, unnormalised output) form
 * of the merge is [SP-CP-survey] section 3.2.
 *
 *   Every query tile of virtual rank r walks the KV chunks that rank holds at
 *   steps 0, 1, ..., P-1 (src = (r - t) mod P), in that order, evaluating the
 *   same (query chunk, held KV chunk) blocks as the per-step ring; instead of
 *   writing each step's (out, lse) and merging it into an accumulator, it
 *   carries the running max, sum and unnormalised output from one step to
 *   the next on chip and writes (out, lse) once.  The result equals
 *   cp_ring_forward_steps' up to rounding (the same terms merged in another
 *   grouping).  Striped: the tile of stripe r walks stripes r, r-1, ...,
 *   each a causal prefix in stripe indices (key i visible to query i' when
 *   i + (stripe > r) <= i').  bf16 inputs (D = 128), any layout (fp32
 *   inputs return CP_ERR_DTYPE); any S the layout allows, 1 <= P <=
 *   CP_MAX_RANKS; no workspace.  Arguments otherwise as cp_ring_forward,
 *   which takes this path for those inputs.
 */
int cp_ring_forward_fused(const void* q, const void* k, const void* v, cp_dtype in_dt,
                          int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                          void* out, cp_dtype out_dt, float* lse, cp_stream_t stream);

/*
 * cp_ring_forward_noalloc - cp_ring_forward for callers that cannot
 * allocate device memory.  The handbook pages have no counterpart: this is a
 * deployment variant of the library, not part of the method.
 *
 *   Who needs it: code that must live inside a fixed device-memory budget
 *   handed out by a host framework (an engine plugin that may not call
 *   cudaMalloc), or code on a latency-critical path where cudaMalloc /
 *   cudaFree would synchronise the device and stall other streams.
 *
 *   Same arguments, layout and results as cp_ring_forward, minus the
 *   workspace.  When cp_ring_forward runs the ring step by step (fp32
 *   inputs) with out_dt = CP_BF16, the fp32
 *   accumulator lives in a 64 MiB array inside the library (static device
 *   memory every GPU that loads the library holds until process exit), so
 *   S*H*D must be <= 16,777,216 (S = 16384 at H = 8, D = 128); larger sizes
 *   return CP_ERR_SHAPE with a message.  With out_dt = CP_F32, or for a ring
 *   cp_ring_forward runs in one launch (bf16 inputs), no scratch is used at
 *   all.  The call allocates nothing.
 *   The first call on a device looks up the array's device address (a
 *   one-time host set-up per device, done with that device current); make
 *   that first call before any stream capture.
 *   Every call on a device shares the one array and it keeps the previous
 *   call's contents; nothing has to start at zero (step 0 writes every
 *   accumulator row before any step reads it), but calls that overlap on the
 *   GPU (different streams, or different host threads) race on it.
 */
int cp_ring_forward_noalloc(const void* q, const void* k, const void* v, cp_dtype in_dt,
                            int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                            void* out, cp_dtype out_dt, float* lse, cp_stream_t stream);

/*
 * cp_ring_step - step t of cp_ring_forward alone (same arguments plus t).
 * Running steps 0..P-1 in order on one stream is cp_ring_forward; between
 * steps (out or workspace, lse) holds the complete ring state, so a caller
 * may stop after step t and resume later.
 */
int cp_ring_step(const void* q, const void* k, const void* v, cp_dtype in_dt,
                 int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                 int step, void* out, cp_dtype out_dt, float* lse,
                 void* workspace, cp_stream_t stream);

/*
 * cp_ring_copy_workspace_size / cp_ring_forward_copy - the ring with its KV
 * physically passed around.  [CP-handbook] section "Ring Attention：KV 沿环
 * 传一圈" and its exercise on overlap (start the transfer of the next block
 * before computing the current one, on a separate stream); [CP-practice]
 * section 7.2 (double-buffered KV so the transfer does not wait for the
 * computation).
 *
 *   Same arguments and result as cp_ring_forward, plus a second stream.
 *   Every virtual rank owns two KV buffers in the workspace.  At step t the
 *   attention launch on `compute_stream` reads rank r's buffer t % 2 (step 0
 *   reads the rank's own rows of k, v in place), while `copy_stream` copies
 *   every rank's held KV into rank r+1's buffer (t+1) % 2 with one
 *   cudaMemcpyAsync per rank and tensor; events order each copy after the
 *   step that last read its destination and each step after the copies it
 *   reads.  The copies only use device memory of this GPU.  The call returns
 *   with all work enqueued; completion is observed on `compute_stream`.
 *   copy_stream may equal compute_stream (no overlap).
 *   workspace: cp_ring_copy_workspace_size() bytes (the fp32 accumulator for
 *   a bf16 output, then the K and V double buffers: 2 * P * R rows each, R =
 *   the rows one rank holds).
 */
int64_t cp_ring_copy_workspace_size(int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                                    cp_dtype in_dt, cp_dtype out_dt);
int cp_ring_forward_copy(const void* q, const void* k, const void* v, cp_dtype in_dt,
                         int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                         void* out, cp_dtype out_dt, float* lse, void* workspace,
                         cp_stream_t compute_stream, cp_stream_t copy_stream);

/*
 * cp_ring_host_workspace_size / cp_ring_forward_host - cp_ring_forward on
 * HOST buffers: the inputs are copied in, the ring runs, and out and lse are
 * copied back, inside one call.  The pages have no counterpart (on a cluster
 * the shards start on their GPUs); this is the entry point for a caller whose
 * sequence lives in host memory.
 *
 *   hq [S,H,D], hk, hv [S,Hkv,D] in in_dt; hout [S,H,D] in out_dt; hlse
 *   [H,S] fp32: HOST memory.  Page-locked memory (cudaHostAlloc /
 *   cudaHostRegister) lets the copies run asynchronously and overlap the
 *   attention; pageable memory gives the same result with the copies
 *   serialised by the driver.
 *   groups: the heads are processed in `groups` groups of H/groups query and
 *   Hkv/groups KV heads (groups must divide Hkv; under GQA group g holds query
 *   heads [g H/groups, (g+1) H/groups) and the KV heads they read).  Heads are
 *   independent, so each group runs the whole ring of cp_ring_forward on its
 *   heads; group g's inputs are copied in on `copy_stream` while group g-1
 *   computes on `stream`, and its results are copied out while group g+1
 *   computes, on a stream the call creates and destroys (so that they do not
 *   queue behind the remaining inputs).  groups = 1: copy in, compute, copy
 *   out, in sequence.
 *   workspace: cp_ring_host_workspace_size() bytes of device memory (staging
 *   for every group's q, k, v, out, lse in compact [S, heads of the group, D]
 *   layout, plus one group's fp32 accumulator for a bf16 output).
 *   The call is ordered after the work already enqueued on `stream` (the
 *   copy stream waits for it) and returns with all work enqueued; `stream`
 *   is made to wait for the last copy, so hout / hlse are complete once
 *   `stream` has completed (e.g. after cudaStreamSynchronize(stream)).
 *   copy_stream may equal stream (no overlap, no extra stream).  Host
 *   buffers must not be written (inputs) or read (outputs) before then.  The
 *   ring's conditions on (S, P, layout) and the dtype rules of
 *   cp_ring_forward apply to each group.  The call creates (and releases)
 *   events and a stream, so it is meant for direct calls, not for capture
 *   into a CUDA graph; the same holds for every *_host entry point below.
 *   Errors: a failure after copies were enqueued (a failed launch) still
 *   makes `stream` wait for every copy the call enqueued before it returns
 *   the error, so after synchronising `stream` no copy touches the host
 *   buffers or the workspace; their contents are then unspecified.  The
 *   same holds for every *_host entry point below.
 */
int64_t cp_ring_host_workspace_size(int64_t S, int H, int Hkv, int D, int groups,
                                    cp_dtype in_dt, cp_dtype out_dt);
int cp_ring_forward_host(const void* hq, const void* hk, const void* hv, cp_dtype in_dt,
                         int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                         void* hout, cp_dtype out_dt, float* hlse, int groups,
                         void* workspace, cp_stream_t stream, cp_stream_t copy_stream);

/*
 * cp_ring_step_blocks - host-only: the blocks the ring evaluates at step t.
 * Writes up to `cap` entries of 4 ints (rank, q_chunk, kv_chunk, diagonal)
 * into `blocks` (host memory) and returns the number of blocks, or a
 * negative cp_status.  Chunks are in the layout's units (P chunks for
 * contiguous, 2P for zigzag, stripes r for striped).  Needs no GPU.
 */
int cp_ring_step_blocks(int P, cp_layout layout, int step, int* blocks, int cap);

/*
 * cp_seq_to_head / cp_head_to_seq - the Ulysses all-to-all on one GPU.
 *   [CP-handbook] section "Ulysses：在序列和头之间转置".
 *
 *   seq_to_head: x [S,H,D] (the P rank shards [S/P,H,D] stacked in rank
 *   order) -> y [P,S,H/P,D] (rank p's [S,H/P,D], stacked):
 *       y[p,s,j,:] = x[s, p*(H/P)+j, :]
 *   head_to_seq: the inverse, y -> x.
 *   dt is the element type (CP_F32 or CP_BF16).  S % P = 0, H % P = 0.
 *   x and y may not overlap.
 */
int cp_seq_to_head(const void* x, void* y, cp_dtype dt, int64_t S, int H,
                   int D, int P, cp_stream_t stream);
int cp_head_to_seq(const void* y, void* x, cp_dtype dt, int64_t S, int H,
                   int D, int P, cp_stream_t stream);

/*
 * cp_ulysses_workspace_size / cp_ulysses_forward - Ulysses attention on one
 * GPU: seq_to_head on q, k, v; causal attention over the full sequence for
 * each rank's head group (H/P query heads, Hkv/P KV heads, offsets 0);
 * head_to_seq on the output.  [CP-handbook] section "Ulysses：在序列和头之间
 * 转置"; the degree is bounded by the KV head count (section "练习"), so
 * Hkv % P = 0 is required.
 *   q [S,H,D], k, v [S,Hkv,D]; out [S,H,D] out_dt; lse [H,S] fp32.
 *   workspace: cp_ulysses_workspace_size() bytes of device memory (holds the
 *   permuted q, k, v and the permuted output).
 */
int64_t cp_ulysses_workspace_size(int64_t S, int H, int Hkv, int D,
                                  cp_dtype in_dt, cp_dtype out_dt);
int cp_ulysses_forward(const void* q, const void* k, const void* v,
                       cp_dtype in_dt, int64_t S, int H, int Hkv, int D, int P,
                       void* out, cp_dtype out_dt, float* lse, void* workspace,
                       cp_stream_t stream);

/*
 * cp_ulysses_host_workspace_size / cp_ulysses_forward_host - the Ulysses
 * forward on HOST buffers.  From host memory the all-to-all is a strided
 * copy: head group p of hq [S,H,D] (rank p's H/P query heads) is copied
 * straight into its own compact [S, H/P, D] block, and likewise for the KV
 * heads it reads, so no permutation kernel runs; each group's causal
 * attention (cp_attn_block over its heads) overlaps the copies of the other
 * groups, and its output goes back into hout [S,H,D] at its heads.
 *   hq [S,H,D], hk, hv [S,Hkv,D] in in_dt; hout [S,H,D] in out_dt; hlse
 *   [H,S] fp32: HOST memory (page-locked for the copies to overlap).  P and
 *   the KV heads as cp_ulysses_forward (P divides H and either divides Hkv or
 *   is a multiple of it; with P > Hkv each group receives its own copy of its
 *   KV head).  workspace: cp_ulysses_host_workspace_size() bytes of device
 *   memory.  Ordering and completion as cp_ring_forward_host.  The result
 *   equals cp_ulysses_forward's.
 */
int64_t cp_ulysses_host_workspace_size(int64_t S, int H, int Hkv, int D, int P, cp_dtype in_dt,
                                       cp_dtype out_dt);
int cp_ulysses_forward_host(const void* hq, const void* hk, const void* hv, cp_dtype in_dt,
                            int64_t S, int H, int Hkv, int D, int P, void* hout, cp_dtype out_dt,
                            float* hlse, void* workspace, cp_stream_t stream,
                            cp_stream_t copy_stream);

/*
 * cp_usp_host_workspace_size / cp_usp_forward_host - cp_usp_forward on HOST
 * buffers: the Ulysses all-to-alls over Pu head groups as strided copies
 * (as cp_ulysses_forward_host), and inside each group the ring of Pr
 * virtual ranks in `layout` of cp_ring_forward, one group's kernels
 * overlapping the other groups' copies.  Arguments as cp_usp_forward with
 * host tensors; workspace: cp_usp_host_workspace_size() bytes of device
 * memory.  Pr >= 1.
 */
int64_t cp_usp_host_workspace_size(int64_t S, int H, int Hkv, int D, int Pu, cp_dtype in_dt,
                                   cp_dtype out_dt);
int cp_usp_forward_host(const void* hq, const void* hk, const void* hv, cp_dtype in_dt,
                        int64_t S, int H, int Hkv, int D, int Pu, int Pr, cp_layout layout,
                        void* hout, cp_dtype out_dt, float* hlse, void* workspace,
                        cp_stream_t stream, cp_stream_t copy_stream);

/*
 * cp_ulysses_stage - one stage of cp_ulysses_forward (same arguments plus
 * `stage`): 0 = seq_to_head of q, k, v into the workspace, 1 = the attention
 * launch over all head groups, 2 = head_to_seq of the output.  Stages 0, 1, 2
 * in order on one stream are cp_ulysses_forward, bit for bit; the workspace
 * carries the state between them.  stage outside [0, 2]: CP_ERR_ARG.
 */
int cp_ulysses_stage(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                     int H, int Hkv, int D, int P, void* out, cp_dtype out_dt, float* lse,
                     void* workspace, int stage, cp_stream_t stream);

/*
 * cp_usp_workspace_size / cp_usp_forward - Ulysses across Pu head groups
 * combined with a ring of Pr virtual ranks inside each group.
 *   [CP-handbook] section "怎么选" (Ulysses inside a node and Ring across
 *   nodes, the USP scheme).  seq_to_head with degree Pu (KV heads replicated
 *   in place when Pu is a multiple of Hkv), then the ring of cp_ring_forward
 *   with Pr ranks and `layout` over each group's whole sequence, then
 *   head_to_seq.  The rings of all Pu groups share each launch: one launch
 *   for the whole ring where cp_ring_forward runs in one (bf16 inputs),
 *   else one per ring step.
 *   The same arguments as cp_ulysses_forward plus Pr and layout; S % Pu = 0
 *   and the ring's own conditions on (S, Pr, layout).
 *   workspace: cp_usp_workspace_size() bytes.
 */
int64_t cp_usp_workspace_size(int64_t S, int H, int Hkv, int D, cp_dtype in_dt,
                              cp_dtype out_dt);
int cp_usp_forward(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                   int H, int Hkv, int D, int Pu, int Pr, cp_layout layout, void* out,
                   cp_dtype out_dt, float* lse, void* workspace, cp_stream_t stream);

/*
 * cp_usp_stage - one stage of cp_usp_forward (same arguments plus `stage`):
 * 0 = seq_to_head of q, k, v, 1 .. Pr = ring step stage-1 (one launch over
 * all Pu groups), Pr + 1 = head_to_seq of the output.  Where the ring runs
 * in one launch (bf16 inputs), stage 1 is the whole
 * ring and stages 2 .. Pr launch nothing.  Stages 0 .. Pr + 1 in order on
 * one stream are cp_usp_forward, bit for bit.  Other stages: CP_ERR_ARG.
 */
int cp_usp_stage(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                 int H, int Hkv, int D, int Pu, int Pr, cp_layout layout, void* out,
                 cp_dtype out_dt, float* lse, void* workspace, int stage, cp_stream_t stream);

/*
 * Backward pass.  The pages time training steps of forward plus backward
 * ([CP-practice] section 4.2) and check that a context-parallel run gives
 * the single-device outputs AND gradients ([SP-CP-survey] section 5.3); they
 * print no backward algorithm.  The gradients below are the chain rule of
 * the forward definition (cp_attn_block), written with the forward's saved
 * whole-row LSE:
 *   p_ij = exp(scale q_i.k_j - lse_i) (0 where masked), delta_i = dO_i . O_i,
 *   dV_j = sum_i p_ij dO_i,  dS_ij = p_ij (dO_i . v_j - delta_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i;
 * under GQA a KV head's gradients sum over the query heads that read it.
 * Inputs q, k, v, out (the forward output) and dout share in_dt: CP_BF16
 * with D = 128 (tensor-core kernels) or CP_F32 with D in {16, 32, 64, 128}
 * (CUDA-core kernels, accurate expf; the toy configuration); gradients are
 * written in grad_dt (CP_F32 or CP_BF16), accumulated in fp32.
 */

/*
 * cp_attn_block_backward - gradients of one block (cp_attn_block's
 * arguments) given the WHOLE-row out and lse: when the block is part of a
 * longer row (a ring step), pass the merged final out / lse, and the block
 * gradients of all blocks of a row add up to the gradients of the row.
 *
 *   q, out, dout [Sq,H,D]; k, v [Sk,Hkv,D]; lse [H,Sq] fp32 (natural log;
 *   -inf = a row that sees no key, its gradients are 0).
 *   dq [Sq,H,D], dk, dv [Sk,Hkv,D] in grad_dt are OVERWRITTEN with this
 *   block's gradients.  workspace: cp_attn_block_backward_workspace_size()
 *   bytes of device memory (delta).  Sq = 0 or Sk = 0 writes zero gradients.
 */
int64_t cp_attn_block_backward_workspace_size(int64_t Sq, int H);
int cp_attn_block_backward(const void* q, const void* k, const void* v, const void* out,
                           const void* dout, const float* lse, cp_dtype in_dt, int64_t Sq,
                           int64_t Sk, int H, int Hkv, int D, int64_t q_offset, int64_t k_offset,
                           int causal, float scale, void* dq, void* dk, void* dv,
                           cp_dtype grad_dt, void* workspace, cp_stream_t stream);

/*
 * cp_ring_backward - gradients of cp_ring_forward (scale 1/sqrt(D)) by the
 * same ring schedule: at step t virtual rank r evaluates the forward's
 * (query chunk, held KV chunk) pairs; dQ of its chunks accumulates in place,
 * dK / dV accumulate on the held chunk (in the ring they travel with it back
 * to their owner).  For bf16 inputs (any layout) one dK/dV launch and one
 * dQ launch cover every step (cp_ring_backward_fused_step), for fp32 inputs
 * one of each per step covers all ranks (cp_ring_backward_step);
 * the blocks use the whole-row lse, so the result equals the gradients of
 * monolithic causal attention up to rounding.
 *
 *   q, out, dout [S,H,D], k, v [S,Hkv,D] in natural order; lse [H,S]
 *   the forward's; layouts and (S, P) conditions as cp_ring_forward.
 *   dq, dk, dv in grad_dt are overwritten.  workspace:
 *   cp_ring_backward_workspace_size() bytes (delta, plus fp32 accumulators
 *   for bf16 gradients).
 */
int64_t cp_ring_backward_workspace_size(int64_t S, int H, int Hkv, int D, cp_dtype grad_dt);

/*
 * cp_ring_backward_step - one launch of the ring backward's per-step
 * schedule, for callers that interleave their own work between launches
 * (in a real ring: sending a chunk's dK / dV on after the step that
 * finished it) and for timing.  launch = -1: the delta preprocessing;
 * launch = 2t: the dK/dV kernel of ring step t, accumulating into the fp32
 * gradient buffers; launch = 2t + 1: the dQ kernel of step t (0 <= t < P).
 * Running launch -1, 0, 1, ..., 2P-1 in order on one stream is the ring
 * backward step by step -- what cp_ring_backward runs for fp32 inputs.
 * Arguments as cp_ring_backward.
 *
 * cp_ring_backward_fused_step - one launch of the two-launch schedule that
 * cp_ring_backward runs for bf16 inputs (fp32 inputs return CP_ERR_DTYPE).
 * launch = -1: delta;
 * launch = 0: the dK/dV kernel over every ring step -- each KV tile stays
 * put while the query chunks that see it stream past in the order the
 * ring's steps bring them to its holder, its dK / dV held in TMEM and
 * written once; launch = 1: the dQ kernel over every step -- each query
 * tile walks the KV chunks its rank holds at steps 0 .. P-1, as the
 * forward's one-launch ring does.  Same gradients as the per-step schedule
 * up to rounding (the same terms summed in another grouping).
 */
int cp_ring_backward_step(const void* q, const void* k, const void* v, const void* out,
                          const void* dout, const float* lse, cp_dtype in_dt, int64_t S, int H,
                          int Hkv, int D, int P, cp_layout layout, int launch, void* dq,
                          void* dk, void* dv, cp_dtype grad_dt, void* workspace,
                          cp_stream_t stream);
int cp_ring_backward_fused_step(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse, cp_dtype in_dt, int64_t S,
                                int H, int Hkv, int D, int P, cp_layout layout, int launch,
                                void* dq, void* dk, void* dv, cp_dtype grad_dt, void* workspace,
                                cp_stream_t stream);
int cp_ring_backward(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, cp_dtype in_dt, int64_t S, int H,
                     int Hkv, int D, int P, cp_layout layout, void* dq, void* dk, void* dv,
                     cp_dtype grad_dt, void* workspace, cp_stream_t stream);

/*
 * cp_ring_backward_host_workspace_size / cp_ring_backward_host -
 * cp_ring_backward on HOST buffers, the counterpart of cp_ring_forward_host:
 * q, k, v, out, dout and lse are copied in, the ring backward runs, and dq,
 * dk, dv are copied back, in `groups` head groups (groups divides Hkv; group g
 * holds query heads [g H/groups, (g+1) H/groups) and the KV heads they read)
 * whose copies on `copy_stream` overlap the other groups' kernels on
 * `stream`.  Heads are independent, so each group runs the whole backward of
 * its heads.
 *   hq, hout, hdout [S,H,D], hk, hv [S,Hkv,D] in in_dt; hlse [H,S] fp32;
 *   hdq [S,H,D], hdk, hdv [S,Hkv,D] in grad_dt: HOST memory (page-locked for
 *   the copies to overlap).  workspace: cp_ring_backward_host_workspace_size()
 *   bytes of device memory (compact per-group staging of every input and
 *   gradient, plus one group's cp_ring_backward workspace).  Ordering and
 *   completion as cp_ring_forward_host: the gradients are in host memory once
 *   `stream` has completed.
 */
int64_t cp_ring_backward_host_workspace_size(int64_t S, int H, int Hkv, int D, int groups,
                                             cp_dtype in_dt, cp_dtype grad_dt);
int cp_ring_backward_host(const void* hq, const void* hk, const void* hv, const void* hout,
                          const void* hdout, const float* hlse, cp_dtype in_dt, int64_t S,
                          int H, int Hkv, int D, int P, cp_layout layout, void* hdq, void* hdk,
                          void* hdv, cp_dtype grad_dt, int groups, void* workspace,
                          cp_stream_t stream, cp_stream_t copy_stream);

/*
 * cp_check_device_error - synchronise `stream`, then report and clear the
 * device status word: CP_OK, or CP_ERR_TIMEOUT if a kernel's bounded wait
 * expired since the last check (the kernel then skipped the rest of its
 * work and its outputs are undefined), CP_ERR_BOUNDS (bounds-checked build
 * only) if a kernel found a tile or row outside its tensor (it skipped
 * those reads and writes; the message names the check), or CP_ERR_CUDA if
 * the synchronisation failed.  The first error since the last check wins.
 */
int cp_check_device_error(cp_stream_t stream);

/*
 * cp_debug_bounds - 1 in the bounds-checked build of the library
 * (libcpattn_debug.so, compiled with CP_DEBUG_BOUNDS), 0 in the release
 * build (libcpattn.so).  In the bounds-checked build every attention kernel
 * (forward and backward, tensor-core and fp32) checks, per tile or row,
 * that what it reads and writes of q, k, v, out / acc, lse, delta and the
 * gradients lies inside the tensors the call describes, records a failure
 * in the device status word (see cp_check_device_error) and skips the
 * access.  Results are otherwise bit-identical to the release build.
 */
int cp_debug_bounds(void);

/*
 * cp_selftest_wait_timeout - failure-detection self-test: launches one
 * block that waits on an mbarrier nothing will complete, with a limit of
 * `timeout_us` microseconds (1..2000000).  The wait expires, the kernel
 * records CP_ERR_TIMEOUT and returns normally; a following
 * cp_check_device_error() reports it.  No fault, trap or hang is involved.
 */
int cp_selftest_wait_timeout(int timeout_us, cp_stream_t stream);

/* Last error message of the calling thread ("" if none). */
const char* cp_last_error(void);

/* Library version string. */
const char* cp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
