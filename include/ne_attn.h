/*
 * ne_attn: causal grouped-query attention with rotary position embedding on
 * Q and K, forward and backward, for NVIDIA GB300 (sm_103a).
 *
 * The operation is the attention block of the NanoEuler decoder-only
 * transformer (socker-news README, "Architecture": rotary embedding applied
 * to queries and keys, grouped-query attention in which query heads share a
 * smaller set of key/value heads; "GPU engine": a tiled FlashAttention with
 * online softmax that never forms the T x T matrix; mynewscn README, same
 * items).  For every batch b, query head h (key/value head g = h / (Hq/Hkv))
 * and position t:
 *
 *   q^_t = R_t q[b,t,h],  k^_j = R_j k[b,j,g]       rotary embedding, interleaved
 *                                                   pairs (2i, 2i+1), angle
 *                                                   t * base^(-2i/D)
 *   s_tj = q^_t . k^_j / sqrt(D)  for j <= t        causal: later keys are skipped
 *   o[b,t,h] = sum_j softmax_j(s_t.) v[b,j,g]
 *   lse[b,h,t] = ln sum_{j<=t} exp(s_tj)            natural log
 *
 * Layouts (row-major, contiguous):
 *   q, o, dout, dq : [B, T, Hq,  D]   bfloat16 (o and dq may be float32, see flags)
 *   k, v, dk, dv   : [B, T, Hkv, D]   bfloat16 (dk, dv may be float32)
 *   lse            : [B, Hq, T]       float32
 * Supported: D in {32, 64}; Hq % Hkv == 0; 1 <= T; B >= 1; and
 * B * T * max(Hq, Hkv) * D < 2^31.  All tensor pointers are device pointers,
 * 16-byte aligned; the caller owns every buffer.
 *
 * Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 * default stream): no host synchronisation, no host<->device copies.  Argument
 * errors are detected on the host and returned before anything is launched.
 * A kernel whose internal pipeline wait exceeds its time limit stops, frees
 * its tensor memory and records NE_ERR_DEVICE_TIMEOUT in a device status word
 * that ne_attn_check_status() reads.
 *
 * The library keeps one small table per (device, D, rope_base): fp32
 * cos/sin of t * theta_i for t below the largest T seen so far, built on the
 * device in double precision; and, per forward shape, the table of work items
 * of each CTA of the persistent forward kernel (built on the host, copied once).
 * The first call that needs a new or larger table allocates it with
 * cudaMalloc, so make one call per shape (with the largest T) before capturing
 * calls in a CUDA graph.  Calls that pass no workspace use a buffer of the
 * library's per stream (see ne_attn_fwd_ex).  Nothing else is allocated.
 */
#ifndef NE_ATTN_H
#define NE_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NE_OK = 0,
  NE_ERR_ARG = -1,            /* null pointer, bad size, Hq % Hkv != 0, bad rope_base or flags */
  NE_ERR_ALIGN = -2,          /* a tensor pointer is not 16-byte aligned */
  NE_ERR_UNSUPPORTED = -3,    /* D not in {32, 64}, size limits, or device is not sm_103 */
  NE_ERR_CUDA = -4,           /* a CUDA runtime/driver call or a launch failed */
  NE_ERR_WORKSPACE = -5,      /* workspace missing, too small or not 256-byte aligned */
  NE_ERR_DEVICE_TIMEOUT = -6, /* a kernel gave up on a pipeline wait (see above) */
  NE_ERR_SCRATCH_LIMIT = -7   /* ne_attn_bwd_noalloc: problem too large for its fixed scratch */
} ne_status;

/* Flag bits for ne_attn_fwd_ex, ne_attn_bwd and the workspace-size queries. */
#define NE_ATTN_O_FP32 1     /* o is float32 [B,T,Hq,D] (forward output, backward input) */
#define NE_ATTN_GRAD_FP32 2  /* dq, dk, dv are float32 */
#define NE_ATTN_PRECISE_QK 4 /* split precision for inputs whose logits reach |s| ~ 10^2..10^4
                                (default precision rounds the rotated q, k to fp16, 2^-11
                                relative, which there moves a logit by whole units: on such
                                inputs its dq and dk are several percent off):
                                S = qhi.khi + qlo.khi + qhi.klo from fp16 hi + lo parts of the
                                rotated q and k (three tensor-core products instead of one);
                                P = Phi + Plo (two bf16 parts) in O += P V and dV += P^T dO;
                                dS = dShi + dSlo (two fp16 parts) in dK and dQ; and lse holds
                                2*B*Hq*T floats: the fp32 LSE [B,Hq,T] followed by its fp32
                                remainder [B,Hq,T] (LSE = hi + lo), which the backward uses to
                                rebuild P where one fp32 ulp of the LSE is already ~1e-3.
                                Use the same setting for the forward and the backward. */
#define NE_ATTN_QK_ROTATED 8 /* default precision: the first ne_attn_fwd_workspace_size bytes
                                of `workspace` hold the rotated q and k (fp16) for these q, k and
                                rope_base, so the call does not rotate them again.  The forward's
                                workspace is laid out as the start of the backward's.
                                ne_attn_fwd_ex: ne_attn_qkv_rmsnorm wrote them there (same flag);
                                the workspace is then required and q, k may be NULL.
                                ne_attn_bwd: ne_attn_fwd_ex or ne_attn_qkv_rmsnorm wrote them.
                                ne_attn_qkv_rmsnorm: write them.  Rejected with
                                NE_ATTN_PRECISE_QK and by ne_attn_bwd_noalloc. */
#define NE_ATTN_ROPE_HALF 16 /* rotary pairs (x[i], x[i + D/2]) (the half-split layout) instead
                                of the interleaved (x[2i], x[2i+1]); same angles t * base^(-2i/D)
                                for pair i.  The pages name no pair layout.  Accepted by the
                                forward, the backward (both calls of a step must agree, as with
                                NE_ATTN_QK_ROTATED), ne_attn_kv_append and ne_attn_decode (the
                                cache and the queries must agree); not with NE_ATTN_PRECISE_QK
                                (NE_ERR_UNSUPPORTED). */
#define NE_ATTN_FP8 32       /* forward only (an inference variant), D = 64, Hq + Hkv <= 256:
                                the rotated q and k are rounded to e4m3 with one scale per head
                                (code = value * 448 / max |value| of the head over the whole
                                batch, round to nearest even) and S = Q K^T runs on the tensor
                                cores' 8-bit path (kind::f8f6f4); v, P and O keep their formats.
                                Expect about 3e-2 relative error in o (the e4m3 rounding of q, k
                                alone); not with NE_ATTN_PRECISE_QK or NE_ATTN_QK_ROTATED
                                (NE_ERR_ARG), other D (NE_ERR_UNSUPPORTED).  The workspace
                                holds the e4m3 q, k and the maxima (ne_attn_fwd_workspace_size
                                with this flag). */

/*
 * Forward pass: writes o (bfloat16) and lse.  Same as ne_attn_fwd_ex with
 * flags = 0 and no workspace.
 * Two kernels.  A streaming pre-pass applies the rotary embedding to q and k
 * and stores the rotated values as fp16 (3 more mantissa bits than bf16) in
 * the workspace.  The attention kernel then runs one CTA per SM over work
 * items (query tile x query heads of one key/value head): K/V tiles are
 * loaded once per key/value head and shared by the query heads of its group;
 * S = Q K^T and O += P V run on the tensor cores (fp32 accumulation in tensor
 * memory; P is bf16) with an online softmax in between.  Returns NE_OK or a
 * negative ne_status.
 */
int ne_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T,
                int Hq, int Hkv, int D, float rope_base, void* stream);

/*
 * Bytes of device workspace the forward needs for this shape and flags: the
 * rotated q [B,T,Hq,D] and k [B,T,Hkv,D] as fp16, each rounded up to 256
 * bytes (0 with NE_ATTN_PRECISE_QK, whose kernel rotates the tiles in shared
 * memory).  The same two arrays start the backward's workspace, at the same
 * offsets.  Returns 0 for unsupported shapes or flags.
 */
size_t ne_attn_fwd_workspace_size(int B, int T, int Hq, int Hkv, int D, int flags);

/*
 * Forward pass with flags (NE_ATTN_O_FP32, NE_ATTN_PRECISE_QK, NE_ATTN_ROPE_HALF,
 * NE_ATTN_QK_ROTATED, NE_ATTN_FP8; others rejected) and an optional caller workspace (256-byte aligned, at least
 * ne_attn_fwd_workspace_size bytes, else NE_ERR_WORKSPACE; the caller owns it
 * and must not touch it until the call's work on `stream` is done).  With
 * workspace = NULL the library uses a buffer of its own per stream, grown
 * with cudaMalloc when a larger shape arrives; while the stream is captured
 * into a CUDA graph it cannot grow and the call returns NE_ERR_WORKSPACE.
 */
int ne_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T,
                   int Hq, int Hkv, int D, float rope_base, int flags, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace ne_attn_bwd needs for this shape and flags
 * (pass a 256-byte aligned pointer).  The pages' backward keeps the softmax
 * statistics of the forward and recomputes the probabilities from them
 * (socker-news README, "Verified backward" and "GPU engine": FlashAttention
 * never stores the T x T matrix); this buffer holds what that recomputation
 * and the dQ accumulation need between the backward's kernels.  Holds: the rotated q and k (fp16, plus
 * their fp16 remainders with NE_ATTN_PRECISE_QK), per-row
 * Delta_t = dO_t . O_t and lse * log2(e) (fp32, rows padded to a multiple of
 * 128), and the fp32 dQ accumulator [B, Hq, Tpad, D].  Returns 0 for
 * unsupported shapes or flags.
 */
size_t ne_attn_bwd_workspace_size(int B, int T, int Hq, int Hkv, int D, int flags);

/*
 * Backward pass: given q, k, v, the forward's o and lse, and the upstream
 * gradient dout (bfloat16), writes dq, dk, dv: the gradients with respect to
 * the un-rotated inputs (the inverse rotation R_t^T is applied on the way
 * out).  The pages hand-write this backward, RoPE and the GQA head sharing
 * included, and check it against central finite differences (socker-news
 * README, "Verified backward"; openai-hub article, hand-written forward and
 * backward):
 *   dV = P^T dO,  dP = dO V^T,  Delta_t = dO_t . O_t,  dS = P o (dP - Delta),
 *   dq = R_t^T (dS k^) / sqrt(D),  dk = R_j^T (dS^T q^) / sqrt(D) summed over
 *   the query heads of each key/value head, with P rebuilt from lse.  flags: NE_ATTN_O_FP32 (o is float32), NE_ATTN_GRAD_FP32 (float32
 * gradients, else bfloat16), NE_ATTN_PRECISE_QK.
 * Three kernels: a pre-pass (Delta = rowsum(dO * O), rotated q/k, zeroed dQ
 * accumulator), a key-tile sweep (dK and dV summed over the query heads of
 * the group inside the kernel, dQ partial products added into the fp32
 * accumulator with bulk tensor reductions), and a dQ epilogue.
 * dQ accumulation order varies between runs, so dq is not bitwise
 * reproducible run to run; o, lse, dk and dv are.
 */
int ne_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv,
                int D, float rope_base, int flags, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * Backward pass for callers that cannot allocate device memory: the same
 * result as ne_attn_bwd (same kernels) with no workspace argument.  Flags:
 * NE_ATTN_O_FP32, NE_ATTN_GRAD_FP32, NE_ATTN_PRECISE_QK, NE_ATTN_ROPE_HALF;
 * NE_ATTN_QK_ROTATED is rejected with NE_ERR_ARG, because the fixed array never
 * holds a forward's rotated q and k (the call always rotates them itself).
 * The NanoEuler pages have no counterpart to this entry point; it exists for
 * callers such as plugins whose host process owns every device allocation,
 * or fixed-memory deployments that forbid allocating after start-up, where a
 * call that grows device memory would fail or break the host's accounting.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Scratch (the workspace of ne_attn_bwd plus the rotary table) comes from one
 * fixed device array of NE_ATTN_STATIC_SCRATCH_BYTES that the library defines;
 * every GPU that loads the library holds it until the process exits.  A
 * problem whose scratch (the ne_attn_bwd_workspace_size figure plus
 * Tpad * D * 4 bytes of table, Tpad = T rounded up to 128) does not fit is
 * rejected with NE_ERR_SCRATCH_LIMIT before anything is launched; the
 * 116M-model shape (B=16, T=512, Hq=12, Hkv=4, D=64) fits.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  Every call uses the same array and it keeps the previous
 * call's contents; the call rebuilds the table and zeroes the accumulator it
 * needs.  Calls whose kernels overlap on the GPU (different streams, or
 * concurrent host threads) race on the array: serialise them.
 */
#define NE_ATTN_STATIC_SCRATCH_BYTES (48u * 1024u * 1024u)
int ne_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv,
                        int D, float rope_base, int flags, void* stream);

/*
 * Incremental decoding with a key/value cache.  The NanoEuler engine generates
 * one token at a time with a KV cache (mynewscn README, generation with the
 * KV cache; socker-news README, GPU generation mode `i`).  A decode step is
 * the forward pass restricted to its newest positions: with Tkv positions in
 * the cache, the Tq new queries sit at positions Tkv - Tq .. Tkv - 1 and
 * o[b,t,h], lse[b,h,t] equal rows Tkv - Tq + t of ne_attn_fwd over T = Tkv.
 *
 * Caches (row-major, head-major, capacity Tcap positions, the caller owns them):
 *   k_cache : [B, Hkv, Tcap, D] fp16, the rotated keys k^_j = R_j k_j
 *   v_cache : [B, Hkv, Tcap, D] bfloat16
 * (head-major so that a decode step reads each head's cache as one stretch)
 *
 * ne_attn_kv_append writes positions pos0 .. pos0 + Tn - 1 of both caches from
 * the new keys and values k_new, v_new [B, Tn, Hkv, D] (bfloat16): each key is
 * rotated at its position and stored as fp16, each value copied.  Requires
 * Tn >= 1, pos0 >= 0, pos0 + Tn <= Tcap.  flags: NE_ATTN_ROPE_HALF or 0.  With
 * NE_ATTN_ROPE_HALF the cached keys hold the rotation in a feature order of the
 * library's own, which only ne_attn_decode with the same flag reads.  One
 * streaming kernel.
 */
int ne_attn_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int B, int Tn,
                      int pos0, int Tcap, int Hkv, int D, float rope_base, int flags, void* stream);

/*
 * Bytes of device workspace ne_attn_decode needs (pass a 256-byte aligned
 * pointer): the rotated queries packed per key/value head ([B, Hkv, 128, D]
 * fp16) and the partial results of up to ceil(Tkv / 128) splits of the cache
 * per key/value head.  Returns 0 for unsupported shapes.
 */
size_t ne_attn_decode_workspace_size(int B, int Tq, int Tkv, int Hq, int Hkv, int D);

/*
 * Decode attention: q [B, Tq, Hq, D] (bfloat16, not rotated; rotated here at
 * positions Tkv - Tq + t) against cache positions 0 .. Tkv - 1.  Writes
 * o [B, Tq, Hq, D] (bfloat16, or float32 with NE_ATTN_O_FP32)
 * and lse [B, Hq, Tq] (flags: NE_ATTN_O_FP32, NE_ATTN_ROPE_HALF as given to
 * ne_attn_kv_append).  Requires 1 <= Tq <= Tkv <= Tcap and
 * (Hq / Hkv) * Tq <= 128: the queries of one key/value head fill at most one
 * 128-row tile, which every K/V tile of the cache serves at once.  The
 * workspace is required.
 * Two kernels: query rotation and packing; a sweep over the cache in which
 * one CTA per SM takes work items (batch, key/value head, split of the key
 * tiles) and runs S = Q K^T and O += P V on the tensor cores with an online
 * softmax, where the CTA that finishes the last split of a (batch, key/value
 * head) merges that group's splits.  The result is bitwise reproducible.
 */
int ne_attn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Tq,
                   int Tkv, int Tcap, int Hq, int Hkv, int D, float rope_base, int flags, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * The step in front of attention: pre-norm RMSNorm and the fused Q/K/V
 * projection without bias (socker-news README, "Architecture" and the block
 * order x = x + attn(rmsnorm(x)); mynewscn README).  For row r = b * T + t:
 *
 *   rstd[r] = 1 / sqrt(mean_c x[r, c]^2 + eps)
 *   qkv[r, n] = sum_c x[r, c] * rstd[r] * norm_w[c] * w_qkv[n, c]
 *   q[b,t,h,:] = qkv[r, h*D ..],  k[b,t,g,:] = qkv[r, Hq*D + g*D ..],
 *   v[b,t,g,:] = qkv[r, (Hq+Hkv)*D + g*D ..]
 *
 * x [B, T, C], norm_w [C] and w_qkv [(Hq + 2 Hkv) D, C] (output by input) are
 * bfloat16; q [B,T,Hq,D], k and v [B,T,Hkv,D] are bfloat16 outputs; rstd
 * [B*T] float32 is an output (the RMSNorm backward needs it).  Requires
 * C % 8 == 0 and the attention shape rules above.  eps > 0.
 * flags: NE_ATTN_QK_ROTATED also writes the rotated q and k (rotary embedding
 * at position t, as ne_attn_fwd applies it) as fp16 into the first
 * ne_attn_fwd_workspace_size bytes of `workspace`, where ne_attn_fwd_ex and
 * ne_attn_bwd with NE_ATTN_QK_ROTATED (and the same workspace, rope_base and
 * rotary layout) take them; q and k may then be NULL.  NE_ATTN_ROPE_HALF
 * selects the half-split rotary pairs for those.  The workspace
 * (ne_attn_qkv_workspace_size bytes, 256-byte aligned) is required with
 * NE_ATTN_QK_ROTATED; with workspace = NULL otherwise the library uses its
 * per-stream buffer as ne_attn_fwd_ex does.
 * Two kernels: per-row rstd together with the projection matrix scaled by
 * norm_w (bf16, in the workspace); then a persistent tensor-core GEMM over
 * 128-row tiles whose epilogue applies rstd and the rotation and stores.
 */
size_t ne_attn_qkv_workspace_size(int B, int T, int C, int Hq, int Hkv, int D, int flags);
int ne_attn_qkv_rmsnorm(const void* x, const void* norm_w, const void* w_qkv, void* q, void* k, void* v,
                        float* rstd, int B, int T, int C, int Hq, int Hkv, int D, float eps, float rope_base,
                        int flags, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: NE_OK, NE_ERR_DEVICE_TIMEOUT, or NE_ERR_CUDA if the
 * synchronisation itself failed.  The pages have no counterpart to this
 * call; it reports the one failure the kernels detect themselves, a pipeline
 * wait that gave up, while the GPU context stays usable.
 */
int ne_attn_check_status(void* stream);

/* Static description of a status code. */
const char* ne_attn_status_string(int status);

/*
 * Kernel timing.  Between ne_attn_profile_start(capacity) and
 * ne_attn_profile_stop(), each kernel that the library's calls launch is
 * bracketed by a pair of CUDA timing events recorded on the launch
 * stream (at most `capacity` launches; later ones are not timed but still
 * counted).  ne_attn_profile_stop synchronises those events and fills, per
 * kernel kind (NE_ATTN_KERNEL_*), the summed device time in milliseconds and
 * the number of launches; arrays must hold NE_ATTN_NUM_KERNEL_KINDS entries.
 * Starting while a profile is open discards it.  Returns NE_OK or a negative
 * ne_status.
 *
 * Calls made while a stream is captured into a CUDA graph record their events
 * into the graph, so the events are re-recorded each time the graph runs.  For
 * that use, ne_attn_profile_detach() ends recording and keeps the events;
 * ne_attn_profile_read() then returns, per kind, the device time and the count
 * of timed launches of the most recent run, as often as needed, until the next
 * ne_attn_profile_start.
 */
#define NE_ATTN_KERNEL_FWD 0
#define NE_ATTN_KERNEL_BWD_PREP 1
#define NE_ATTN_KERNEL_BWD_DKDV 2
#define NE_ATTN_KERNEL_BWD_DQ 3
#define NE_ATTN_KERNEL_FWD_ROPE 4 /* the forward's RoPE pre-pass */
#define NE_ATTN_KERNEL_KV_APPEND 5
#define NE_ATTN_KERNEL_DECODE 6     /* the split sweep over the cache */
#define NE_ATTN_KERNEL_DECODE_AUX 7 /* query rotation and packing */
#define NE_ATTN_KERNEL_QKV_PREP 8   /* RMSNorm row statistics and the weight fold */
#define NE_ATTN_KERNEL_QKV 9        /* the projection GEMM with the rotary epilogue */
#define NE_ATTN_NUM_KERNEL_KINDS 10
int ne_attn_profile_start(int capacity);
int ne_attn_profile_stop(double* total_ms, long long* launches);
int ne_attn_profile_detach(void);
int ne_attn_profile_read(double* total_ms, long long* launches);

/*
 * Test hook for the timeout path: launches one block that waits on a
 * barrier nothing will complete, with the given limit in microseconds
 * (1..1000000), then records NE_ERR_DEVICE_TIMEOUT exactly as the attention
 * kernels do.  Returns NE_OK if the launch succeeded.
 */
int ne_attn_debug_timeout_probe(int limit_us, void* stream);

/*
 * Host-only view of the persistent forward's work schedule (no device call)
 * for B batches, Hkv key/value heads of G query heads each, nt query tiles and
 * nsm SMs.  A work item pairs two units (query head, 128-row query tile) of one
 * (batch, key/value head) that share the item's key/value tiles; each of the
 * kernel's two softmax warpgroups owns one unit.  Writes *grid = min(items,
 * nsm), *K (items of the busiest CTA) and the [grid, K] table of int4 entries
 * (b, h0 | (h1 + 1) << 16, i0, i1) into `table` (4 ints per entry; h1 + 1 = 0
 * for an item of one unit; b = -1 pads a CTA's row).  NE_ERR_ARG (with *grid
 * and *K set) if capacity < 4 * grid * K.
 */
int ne_attn_debug_fwd_schedule(int B, int Hkv, int G, int nt, int nsm, int* table, int capacity, int* grid,
                               int* K);

#ifdef __cplusplus
}
#endif

#endif /* NE_ATTN_H */
