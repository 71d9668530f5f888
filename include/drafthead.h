/*
 * drafthead.h -- C ABI of the GB300 (sm_103a) low-bit speculative-decoding draft head.
 *
 * The operation is the draft head of the page "radiance_drafthead.py" (its module docstring;
 * its load-time quantiser, int2 coarse kernel, block candidate emission, exact rerank and head
 * application):
 *   logits = x[M, K] @ W^T for a vocabulary head W[N, K] (vocab rows, the lm_head layout),
 * computed coarsely from int2 (or int4) codes with an asymmetric per-(vocab row, group of G
 * along K) scale and zero point, after which each 64-row block keeps its KCAND largest coarse
 * values, the RERANK largest of those are rescored exactly against the bf16 weight, and the
 * argmax of the rescored logits is returned per hidden row.
 *
 * Conventions (every entry point):
 *  - All tensor arguments are DEVICE pointers owned by the caller; the library allocates no
 *    device memory and keeps no tensors. Inputs are never written.
 *  - bf16 tensors are passed as `void*` / `const void*` and hold IEEE bfloat16 bit patterns.
 *  - Every layout is dense row-major with the stated shape (no strides).
 *  - Calls are asynchronous and stream-ordered on `s` (NULL = the legacy default stream). The
 *    return value reports argument validation and launch errors only (cudaGetLastError is read
 *    without synchronising); failures detected inside a kernel are recorded in the workspace
 *    status word (see dh_workspace_status). No call allocates device memory, and none but
 *    dh_workspace_status and dh_draft_head_host synchronises, so the per-call device entry
 *    points can be captured in a CUDA graph.
 *  - On any non-OK return nothing was launched; dh_last_error() gives a message.
 *  - Pointers read with 16-byte vector loads must be 16-byte aligned (DH_ERR_ALIGN otherwise).
 */
#ifndef DRAFTHEAD_H_
#define DRAFTHEAD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dh_stream_t; /* the same handle as cudaStream_t */

#define DH_BLOCK_ROWS 64   /* BLOCK_N of the page: vocab rows per candidate block */
#define DH_MAX_KCAND 64    /* candidates kept per block (at most the block width) */
#define DH_MAX_RERANK 256  /* largest RERANK accepted */
#define DH_MAX_TOKENS 4096 /* largest M accepted */

enum {
  DH_OK = 0,
  DH_ERR_NULL = -1,      /* a required pointer is NULL */
  DH_ERR_SHAPE = -2,     /* sizes out of range or not divisible as required */
  DH_ERR_ALIGN = -3,     /* a pointer is not aligned as required */
  DH_ERR_PARAM = -4,     /* G, bits, kcand or rerank not supported */
  DH_ERR_WORKSPACE = -5, /* workspace NULL, misaligned or smaller than dh_workspace_bytes */
  DH_ERR_CUDA = -6,      /* a CUDA runtime call or a launch failed */
  DH_ERR_DEVICE = -7     /* returned by dh_workspace_status when a kernel flagged a failure */
};

/* Bits of the workspace status word (set by kernels, never cleared by the library). */
#define DH_DEV_WAIT_TIMEOUT 0x1u /* a bounded wait inside the coarse kernel ran out; outputs invalid */
#define DH_DEV_BAD_ID 0x2u       /* the rerank met a candidate id >= N; that slot scored -inf */

/*
 * Offline quantise + pack, int2 (page "radiance_drafthead.py", the load-time quantiser at
 * two bits; module docstring on the quarter-split packing and the hoisted bit-pattern dequant).
 *   W       bf16 [N, K], the head weight, vocab rows.                              (16-B aligned)
 *   G       group size along K: 64 or 128.  Requires K % (4*G) == 0.
 *   packed  u8 [N, K/4] out: byte j of row n = q[j] | q[Q+j]<<2 | q[2Q+j]<<4 | q[3Q+j]<<6, Q=K/4.
 *   S       bf16 [N, K/G] out: bf16(4*sc).
 *   ZS      bf16 [N, K/G] out: bf16(4*sc + zp*sc).
 * with, per (row, group): sc = max((hi-lo)/3, 1e-8), zp = clamp(round(-lo/sc), 0, 3),
 * q = clamp(round(w/sc + zp), 0, 3) in IEEE fp32 (round = half to even).
 */
int dh_quantize_pack_int2(const void* W, int64_t N, int64_t K, int G, uint8_t* packed, void* S,
                          void* ZS, dh_stream_t s);

/*
 * The 4-bit comparison variant ("as in the 4-bit path"; packing q[:, :K/2] | q[:, K/2:] << 4,
 * premultiplier 16): requires K % (2*G) == 0; packed u8 [N, K/2]; S = bf16(16 sc),
 * ZS = bf16(16 sc + zp sc); codes 0..15.
 */
int dh_quantize_pack_int4(const void* W, int64_t N, int64_t K, int G, uint8_t* packed, void* S,
                          void* ZS, dh_stream_t s);

/*
 * The int2 quantiser on an FP8 head (the load-time quantiser applied to the head's e4m3 rows
 * with their per-row scale, the page's per-channel FP8 lm_head): the values quantised are
 * fp32(e4m3(W8[n, k])) * row_scale[n] (one fp32 multiply), then exactly as
 * dh_quantize_pack_int2.
 *   W8         e4m3 [N, K] row bytes (e4m3 decoded bit-exactly: no NaN handling).   (16-B aligned)
 *   row_scale  fp32 [N].
 */
int dh_quantize_pack_int2_fp8(const uint8_t* W8, const float* row_scale, int64_t N, int64_t K,
                              int G, uint8_t* packed, void* S, void* ZS, dh_stream_t s);

/* Bytes of packed + S + ZS for one head (0 for unsupported arguments). For N=124160, K=5120,
 * G=128, bits=2 this is 178,790,400 (the page's 0.167 GiB/rank). */
size_t dh_packed_bytes(int64_t N, int64_t K, int G, int bits);

/* Workspace bytes the per-call entry points need for these sizes (one workspace serves them
 * all). The workspace must be zero-filled once before first use; calls sharing a workspace
 * must be ordered on one stream. The rerank needs the 256-byte header (status word) only. The
 * coarse pass of more than 16 hidden rows of an int2 head (its tensor-core path) also keeps its
 * scratch after the header: the hidden states laid out as the MMA operand (80 * K * 2 bytes),
 * their group sums and scales, and the per-CTA buffers of coarse keys the block selection reads
 * (256 * 128 * 80 * 4 bytes). */
size_t dh_workspace_bytes(int64_t M, int64_t N, int64_t K, int kcand, int rerank);

/*
 * Coarse pass + block top-KCAND (the page's int2 coarse kernel and its block candidate
 * emission).
 *   x         bf16 [M, K] hidden states, 1 <= M <= DH_MAX_TOKENS.                  (16-B aligned)
 *   packed,S,ZS  as written by dh_quantize_pack_int2 (bits=2) or _int4 (bits=4).  (16-B aligned)
 *   G         64 or 128; requires K % (8*G) == 0 and K <= 5120.
 *   kcand     1..DH_MAX_KCAND candidates per 64-row block.
 *   cand_val  f32 [M, nblk*kcand] out, nblk = ceil(N/64): for hidden row m and block b,
 *             slots b*kcand .. b*kcand+kcand-1 hold the kcand largest coarse values
 *             c[m, n] = sum_g ( S[n,g] * sum_{k in g} x[m,k] (1 + v[n,k]/beta) - ZS[n,g] * sum_{k in g} x[m,k] )
 *             (beta = 4 for int2, 16 for int4), descending, equal values by ascending row id;
 *             slots past the block's last valid row hold (-inf, -1).
 *   cand_id   i32 [M, nblk*kcand] out: the vocab row of each slot.
 *   y_coarse  bf16 [M, N] out or NULL: bf16(c), the coarse logits.
 *   workspace device buffer of ws_bytes >= dh_workspace_bytes(M, N, K, ...), 256-B aligned.
 * Up to 16 hidden rows (and every int4 call) run on warp-level MMAs in passes of 8 rows; more
 * than 16 rows of an int2 head run on the 5th-generation tensor cores in passes of up to 80.
 * The kernels are launched as programmatic dependents: while the preceding kernel in the stream
 * finishes (if it lets its dependents start early, as this library's rerank does) they only warm
 * the L2 cache with the first weight tiles; every read of an input into the SMs, and every
 * output write, happens after that kernel has completed and its writes are visible. So any
 * kernel may produce x, packed, S or ZS directly before this call.
 */
int dh_draft_head_coarse_topk(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                              const void* S, const void* ZS, int64_t N, int G, int bits,
                              int kcand, float* cand_val, int32_t* cand_id, void* y_coarse,
                              void* workspace, size_t ws_bytes, dh_stream_t s);

/*
 * Global top-RERANK over the block candidates, exact rerank, argmax (the page's head
 * application after the coarse pass: the RERANK best candidates, their exact bf16 rescoring,
 * then the caller's argmax).
 *   x         bf16 [M, K] (the same hidden states).                                (16-B aligned)
 *   W         bf16 [N, K] the exact head weight.                                   (16-B aligned)
 *   cand_val, cand_id  f32 / i32 [M, ncand] (any candidate list; ncand >= rerank).
 *   rerank    1..DH_MAX_RERANK.
 *   rr_id     i32 [M, rerank] out: the rerank largest candidates, ordered by candidate value
 *             descending then id ascending (one entry per candidate slot).
 *   rr_logit  f32 [M, rerank] out: sum_k x[m,k] W[rr_id,k] accumulated in fp32 (-inf for an
 *             id < 0; an id >= N also scores -inf and sets DH_DEV_BAD_ID).
 *   argmax_id i32 [M] out: the rr_id with the largest rr_logit, equal logits by lowest id
 *             (-1 when every slot is empty).
 *   y_coarse  bf16 [M, N] in/out or NULL: when given, y[m, rr_id] = bf16(rr_logit) (the
 *             page's scatter of the exact values over the coarse logits).
 *   workspace as for the coarse call.
 */
int dh_draft_head_rerank_argmax(const void* x, int64_t M, int64_t K, const void* W, int64_t N,
                                const float* cand_val, const int32_t* cand_id, int64_t ncand,
                                int rerank, int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                                void* y_coarse, void* workspace, size_t ws_bytes, dh_stream_t s);

/*
 * The whole device-side call (the page's head application from hidden states to the argmax):
 * dh_draft_head_coarse_topk followed by dh_draft_head_rerank_argmax on the same stream, with
 * the arguments and outputs of the two calls (ncand = ceil(N/64) * kcand; y_coarse, when given,
 * holds the coarse logits with the reranked entries scattered over them) and bit-identical
 * results. The arguments of both are validated before anything is launched, and the rerank's
 * kernel starts as a programmatic dependent of the coarse pass.
 *   workspace: ws_bytes >= dh_workspace_bytes(M, N, K, kcand, rerank), zero-filled before its
 *   first use.
 */
int dh_draft_head_argmax(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                         const void* S, const void* ZS, const void* W, int64_t N, int G, int bits,
                         int kcand, int rerank, float* cand_val, int32_t* cand_id, int32_t* rr_id,
                         float* rr_logit, int32_t* argmax_id, void* y_coarse, void* workspace,
                         size_t ws_bytes, dh_stream_t s);

/*
 * Rerank + argmax without a caller workspace. The page has no counterpart to this entry point:
 * it is for callers that cannot allocate device memory -- a plug-in handed only its input and
 * output buffers, code running inside another framework's memory pool or allocator, or a
 * caller whose allocator must not be entered at call time -- and so cannot provide the
 * workspace that dh_draft_head_rerank_argmax takes.
 *   Arguments, outputs and results are those of dh_draft_head_rerank_argmax (same kernels).
 *   Workspace: a fixed array of DH_NOALLOC_SCRATCH_BYTES among the library's device globals;
 *     every device that loads the library holds it until the process exits. The rerank's
 *     workspace is the 256-byte status header whatever the sizes, so every call that passes
 *     the argument checks fits; sizes out of range (M > DH_MAX_TOKENS, K > 32768, ncand > 2^20,
 *     rerank > DH_MAX_RERANK, ...) are rejected with DH_ERR_SHAPE or DH_ERR_PARAM and a
 *     message, before anything is enqueued, by the checks of dh_draft_head_rerank_argmax.
 *   Set-up: the first call on a device, with that device current, looks up the array's device
 *     address (cudaGetSymbolAddress) and keeps it; make that first call before any stream
 *     capture on that device.
 *   Each call that passes the checks clears the part of the array it uses (cudaMemsetAsync on
 *     s) and then launches; nothing is allocated or freed.
 *   All calls on a device share the one array and it keeps the last call's contents: calls
 *     that overlap on the GPU (different streams without ordering between them) race on it and
 *     give wrong results. Order them on one stream.
 *   The device status word lives in the shared array and is not reported: an id >= N still
 *     scores -inf, but DH_DEV_BAD_ID cannot be read back.
 */
#define DH_NOALLOC_SCRATCH_BYTES (1u << 20) /* 1 MiB per device */
int dh_draft_head_rerank_argmax_noalloc(const void* x, int64_t M, int64_t K, const void* W,
                                        int64_t N, const float* cand_val, const int32_t* cand_id,
                                        int64_t ncand, int rerank, int32_t* rr_id,
                                        float* rr_logit, int32_t* argmax_id, void* y_coarse,
                                        dh_stream_t s);

/*
 * dh_draft_head_rerank_argmax against FP8 rows (the page's exact rerank on its FP8 head): the
 * exact logit is
 * sum_k x[m, k] * e4m3(W8[n, k]) * row_scale[n], the e4m3 bytes decoded bit-exactly; fp32
 * accumulation, the row scale applied to the sum. Every other argument and output as there.
 */
int dh_draft_head_rerank_argmax_fp8(const void* x, int64_t M, int64_t K, const uint8_t* W8,
                                    const float* row_scale, int64_t N, const float* cand_val,
                                    const int32_t* cand_id, int64_t ncand, int rerank,
                                    int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                                    void* y_coarse, void* workspace, size_t ws_bytes,
                                    dh_stream_t s);

/*
 * Logits for a top-K caller (the page's top-K-only output: every logit -inf, then the
 * rerank's scatter): y [M, N] bf16 out = -inf everywhere except y[m, rr_id[m, j]] =
 * bf16(rr_logit[m, j]) (round to nearest even), so that a top-K request draws from exactly the
 * RERANK reranked entries. rr_id, rr_logit [M, rerank] as written by
 * dh_draft_head_rerank_argmax; ids outside [0, N) are skipped. Asynchronous on s.
 */
int dh_topk_only_logits(const int32_t* rr_id, const float* rr_logit, int64_t M, int rerank,
                        int64_t N, void* y, dh_stream_t s);

/*
 * Vocabulary-sharded argmax merge (the page's head is "per rank" one vocab shard of the lm_head:
 * module docstring, and the launch-geometry notes timing one rank's 124160-row shard). The vocab
 * rows are split across ranks at multiples of DH_BLOCK_ROWS, so no candidate block straddles two
 * shards; each rank runs the path on its rows (packed, S, ZS and W are row slices; candidate and
 * rr ids are shard-local) and the ranks exchange one 64-bit key per hidden row:
 *   key = (order-preserving bits of the logit) << 32 | (0xFFFFFFFF - global id), top bit flipped,
 * so that the largest signed key over all shards is the global argmax, equal logits going to the
 * lowest vocab id, and a MAX all-reduce of int64 (NCCL or gloo) is the whole exchange.
 *
 * dh_argmax_shard_keys: keys [M] int64 out = the key of the best (logit, id + id_offset) among
 *   the rerank slots of each row (rr_id, rr_logit [M, rerank] as written by the rerank; slots with
 *   an id < 0 are skipped; a row with none gets INT64_MIN). id_offset: the shard's first vocab
 *   row, 0 .. 2^31 - 1. Device arrays, asynchronous on s.
 * dh_argmax_merge: keys [P, M] int64 (P shards' keys, e.g. gathered; P = 1 for keys a MAX
 *   all-reduce already combined) -> argmax_id [M] (global vocab id, -1 if no candidate) and, if
 *   logit is not NULL, logit [M] (that id's reranked logit, -inf if none). Device arrays.
 * The _host variants take host arrays and run on the calling thread (no GPU needed).
 */
int dh_argmax_shard_keys(const int32_t* rr_id, const float* rr_logit, int64_t M, int rerank,
                         int64_t id_offset, int64_t* keys, dh_stream_t s);
int dh_argmax_merge(const int64_t* keys, int P, int64_t M, int32_t* argmax_id, float* logit,
                    dh_stream_t s);
int dh_argmax_shard_keys_host(const int32_t* rr_id, const float* rr_logit, int64_t M, int rerank,
                              int64_t id_offset, int64_t* keys);
int dh_argmax_merge_host(const int64_t* keys, int P, int64_t M, int32_t* argmax_id,
                         float* logit);

/*
 * The whole call from and to host memory (the page's head application end to end): copies x_host (bf16
 * [M, K]) into x_dev, runs dh_draft_head_argmax, copies
 * argmax [M], rr_id [M, rerank] and rr_logit [M, rerank] back into argmax_host, rr_id_host and
 * rr_logit_host, and synchronises (the one call besides dh_workspace_status that does).
 * x_host and the three host arrays must be page-locked (pinned) memory.
 *   x_dev, cand_val, cand_id, rr_id, rr_logit, argmax_id, workspace: device buffers as for
 *   dh_draft_head_argmax (its device outputs are written too); the other arguments likewise.
 * The sequence is captured into a CUDA graph the first time an argument set is seen on a
 * device (on a stream of the library's own) and replayed on s on later calls. When the four
 * host arrays are mapped into the device's address space (page-locked memory on a system with
 * unified addressing, as cudaHostAlloc gives), a copy kernel stages x (the coarse pass starts
 * during it) and the rerank kernel writes the three results into the host arrays directly, so
 * the graph holds kernels only; otherwise it copies with the copy engines. The library
 * keeps the 16 most recent such graphs and one capture stream per device, no device memory. Returns DH_ERR_PARAM while s is being captured; otherwise the first failing step's
 * status. A kernel-side failure is read with dh_workspace_status.
 */
int dh_draft_head_host(const void* x_host, int64_t M, int64_t K, void* x_dev,
                       const uint8_t* packed, const void* S, const void* ZS, const void* W,
                       int64_t N, int G, int bits, int kcand, int rerank, float* cand_val,
                       int32_t* cand_id, int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                       int32_t* argmax_host, int32_t* rr_id_host, float* rr_logit_host,
                       void* workspace, size_t ws_bytes, dh_stream_t s);

/*
 * A host-memory call prepared once (the page's head application end to end, as
 * dh_draft_head_host): dh_host_plan_create validates the arguments of
 * dh_draft_head_host (all but the stream) and captures the call into a CUDA graph that the plan
 * owns (on the current device); dh_host_plan_run replays it on s and synchronises s, so that a
 * repeated call passes two arguments instead of twenty-four. The buffers stay bound to the plan:
 * write the next x into the same x_host, read the results from the same host arrays.
 *   dh_host_plan_create: *plan = NULL on failure (the first failing check's status, as for
 *     dh_draft_head_host); the library keeps no reference to the plan.
 *   dh_host_plan_run: DH_ERR_NULL for a NULL plan, DH_ERR_PARAM while s is being captured;
 *     run it with the device current that the plan was created on.
 *   dh_host_plan_destroy: frees the plan and its graph (NULL is ignored); not while it runs.
 */
typedef struct dh_host_plan_s* dh_host_plan;
int dh_host_plan_create(const void* x_host, int64_t M, int64_t K, void* x_dev,
                        const uint8_t* packed, const void* S, const void* ZS, const void* W,
                        int64_t N, int G, int bits, int kcand, int rerank, float* cand_val,
                        int32_t* cand_id, int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                        int32_t* argmax_host, int32_t* rr_id_host, float* rr_logit_host,
                        void* workspace, size_t ws_bytes, dh_host_plan* plan);
int dh_host_plan_run(dh_host_plan plan, dh_stream_t s);
void dh_host_plan_destroy(dh_host_plan plan);

/*
 * Synchronises `s`, copies the workspace status word to *device_status and returns DH_OK if
 * it is zero, DH_ERR_DEVICE otherwise (DH_ERR_CUDA if the copy fails). The word is sticky:
 * zero the workspace to clear it.
 */
int dh_workspace_status(const void* workspace, size_t ws_bytes, uint32_t* device_status,
                        dh_stream_t s);

/* Message for the last non-OK status returned on the calling host thread ("" if none). */
const char* dh_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DRAFTHEAD_H_ */
