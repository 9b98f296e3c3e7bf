/*
 * swa_attn.h -- C ABI of the GB300 (sm_103a) causal / sliding-window
 * grouped-query attention library: forward with per-row logsumexp, and an
 * O(L*D)-memory backward that never forms the L x L score matrix and skips
 * every key tile outside the causal / window band.
 *
 * The operation (page "Lab 028 lab detail: Off NVIDIA, you fix the platform
 * yourself", sections "Plan for the build" step 4 and "What I changed, in
 * plain terms" items 1-5; page "Training -- design (ORPO, flash-CCE head,
 * prefix sharing, segmented backward)" sections 5.2 and 6):
 *
 *   band(i) = { j : j <= i  and  (window == 0  or  i - j < window) }
 *   s_ij    = scale * q_i . k_j              (j in band(i))
 *   lse_i   = ln sum_{j in band(i)} exp(s_ij)
 *   o_i     = sum_{j in band(i)} exp(s_ij - lse_i) v_j
 *
 * window == 0 means plain causal; window >= L is the same as causal.  A key
 * that is window or more positions behind the query is masked ("zero P where
 * j < i + diag_off - window_size + 1", diag_off = 0 here: queries and keys
 * have the same length L).  Query head h reads kv head h / (Hq / Hkv)
 * (page "MiniCPM5 Decode Megakernel -- end-to-end build plan", section 4.1
 * stage 5).
 *
 * Conventions shared by every entry point
 *  - Tensors are dense row-major [B, H, L, D]; lse is [B, Hq, L].
 *  - q, k, v, dO hold bf16 values (raw 16-bit patterns, swa_bf16).
 *    o, lse, dq, dk, dv are fp32.
 *  - All tensor and workspace pointers are DEVICE pointers owned by the
 *    caller.  The library allocates no device or host memory on these
 *    paths.  Every output is fully overwritten (no accumulate-into).
 *  - The first swa_attn_bwd / swa_attn_bwd_ex call on a device creates one
 *    CUDA stream (highest priority, non-blocking) and two events for that
 *    device, kept until the process exits; make that first call outside
 *    stream capture.  Each backward runs its dK/dV pass on that stream,
 *    beside the dQ pass on `stream`: the internal stream waits for the work
 *    already on `stream`, and `stream` waits for the dK/dV pass before the
 *    call returns.  Everything a call enqueues is therefore ordered on
 *    `stream` as one sequence, and a call captured into a CUDA graph from
 *    `stream` captures both passes.
 *  - Tensor pointers must be 16-byte aligned; the workspace 256-byte aligned.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) of the current device, which must be an sm_103
 *    GPU.  Return values report argument and launch errors only: SWA_OK
 *    says the work was enqueued, not that it succeeded.  Failures detected
 *    on the device are latched in a per-device status word read by
 *    swa_attn_get_status(): a bounded wait that ran out
 *    (SWA_ERR_DEVICE_TIMEOUT), an input that overflowed an fp16 operand copy
 *    (SWA_ERR_FP16_RANGE), an SM id outside the head-dim-512 scratch
 *    (SWA_ERR_SCRATCH_LAYOUT).  The outputs of such a call are undefined
 *    (they may hold inf or NaN); poll the status to detect it.
 *  - Operand precision.  The tensor cores multiply fp16 copies of the bf16
 *    inputs, with fp32 accumulation; S and dP stay fp32, P and
 *    dS = P (dP - Delta) are rounded to fp16.  The copies are exact for
 *    2^-14 <= |x| < 65504.  The forward copies v; the backward copies q, k,
 *    v and dO.  A q, k or v entry of magnitude 65504 or more latches
 *    SWA_ERR_FP16_RANGE; entries below 2^-14 lose precision (fp16
 *    subnormals).  dO is different: the backward scales its copy by a power
 *    of two s chosen from max |dO| (the scaled maximum lies in [4, 8)), keeps
 *    Delta scaled the same way and multiplies dq, dk and dv by 1/s at the
 *    end, all exactly.  So any finite dO works, tiny cotangents keep their
 *    precision, and scaling dO by a power of two scales dq, dk and dv by the
 *    same power bit for bit.
 *  - Supported head dims: 64, 128, 256, 512.  scale is any finite float.
 *  - Head dim 512 hands tiles between the CTAs of a cluster through a static
 *    L2 scratch of the library (36 MB per device) indexed by the receiving
 *    CTA's SM id.  Its kernels fill an SM (one CTA per SM), and SM ids must be
 *    below 192.  The first head-dim-512 call on a device checks both on the
 *    host and returns SWA_ERR_SCRATCH_LAYOUT if the device does not meet
 *    them.
 *  - Thread safety: calls on different streams may overlap if they use
 *    different workspaces.  At head dim 512 this holds because no two CTAs
 *    of these kernels share an SM, so no two share a scratch slot (checked as
 *    above).  swa_attn_bwd_noalloc is the exception: see there.
 */
#ifndef SWA_ATTN_H
#define SWA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t swa_bf16; /* bf16 bit pattern */

/* Return codes (0 = success, negative = error). */
#define SWA_OK 0
#define SWA_ERR_NULL_POINTER -1   /* a required pointer is NULL */
#define SWA_ERR_BAD_SHAPE -2      /* B, Hq, Hkv or L (Lq) < 1, or Lk < Lq */
#define SWA_ERR_BAD_GROUPS -3     /* Hq is not a multiple of Hkv */
#define SWA_ERR_BAD_HEAD_DIM -4   /* D not in {64, 128, 256, 512} */
#define SWA_ERR_BAD_WINDOW -5     /* window < 0 */
#define SWA_ERR_BAD_SCALE -6      /* scale is NaN or infinite */
#define SWA_ERR_MISALIGNED -7     /* tensor not 16-B or workspace not 256-B aligned */
#define SWA_ERR_WORKSPACE -8      /* workspace_bytes below the query's value */
#define SWA_ERR_CUDA -9           /* CUDA runtime / launch error */
#define SWA_ERR_TOO_LARGE -10     /* sizes exceed the supported index range */
#define SWA_ERR_DEVICE_TIMEOUT -11 /* a bounded device-side wait expired */
#define SWA_ERR_UNSUPPORTED_DEVICE -12 /* current device is not sm_103 */
#define SWA_ERR_NOALLOC_LIMIT -13 /* B*Hq*L above swa_attn_bwd_noalloc's fixed scratch */
#define SWA_ERR_FP16_RANGE -14    /* device: an input magnitude overflowed the fp16 operand copy */
#define SWA_ERR_SCRATCH_LAYOUT -15 /* head dim 512: device cannot hold the per-SM tile scratch (see below) */
#define SWA_ERR_BAD_PLAN -16      /* shared-prefix plan: prompt_len or chosen_len out of range */

/*
 * Workspace bytes swa_attn_fwd needs for this shape (may be 0; a NULL
 * workspace is then accepted).  Pure host function, no CUDA calls.
 */
size_t swa_attn_fwd_workspace_bytes(int B, int Hq, int Hkv, int L, int D, int window);

/*
 * Queries that are a suffix of the keys, and non-causal windows
 * ("Lab 028 lab detail", "What I changed, in plain terms" items 3-6 and
 * "Gradient parity": diag_off = kL - qL, windows "causal and not", and
 * zero dK/dV for keys that no query's window reaches).
 *
 * q and dO are [B, Hq, Lq, D], o is [B, Hq, Lq, D], lse [B, Hq, Lq]; k, v,
 * dk and dv are [B, Hkv, Lk, D], with 1 <= Lq <= Lk.  Query row i sits at
 * key position a = i + (Lk - Lq), so Lq = Lk is self-attention and Lq = 1
 * is one decode step over a cache of Lk keys.  The band of row i is
 *
 *   causal != 0:  { j : j <= a  and  (window == 0  or  a - j < window) }
 *   causal == 0:  { j : window == 0  or  |a - j| < window }
 *
 * (causal == 0 with window == 0 is unmasked attention over all Lk keys).
 * Every row sees at least the key at its own position.  Keys that no query
 * sees get dk = dv = 0 exactly.  A window of Lk or more is the same as no
 * window.  Everything else (dtypes, alignment, workspace, streams, status
 * word, errors) is as for swa_attn_fwd / swa_attn_bwd, which are these
 * calls with Lq = Lk = L and causal = 1.  Lk < Lq returns SWA_ERR_BAD_SHAPE.
 */
size_t swa_attn_fwd_workspace_bytes_ex(int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal);
size_t swa_attn_bwd_workspace_bytes_ex(int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal);
int swa_attn_fwd_ex(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, float* o, float* lse,
                    int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal, float scale,
                    void* workspace, size_t workspace_bytes, void* stream);
int swa_attn_bwd_ex(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o,
                    const float* lse, const swa_bf16* dO, float* dq, float* dk, float* dv,
                    int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal, float scale,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Shared prompt prefix ("Training -- design (ORPO, flash-CCE head, prefix
 * sharing, segmented backward)", section 5.4 "Shared prompt-prefix
 * forward"): one causal self-attention pass over a sequence of L rows laid
 * out as [prompt (prompt_len rows); chosen response (chosen_len rows);
 * rejected response (the remaining rows)], in place of two passes over
 * [prompt; chosen] and [prompt; rejected].  The mask is "causal AND NOT
 * rejected -> chosen", and the window is measured on logical positions:
 * each response starts right after the prompt, so with lp(x) = x - chosen_len
 * for rejected rows and lp(x) = x otherwise,
 *
 *   key j visible to query i  iff  j <= i,
 *                                  not (i rejected and j chosen),
 *                                  and (window == 0 or lp(i) - lp(j) < window).
 *
 * A rejected row therefore sees two key intervals (part of the prompt and
 * its own response), and the kernels visit only the key tiles those
 * intervals meet.  The prompt rows are computed once; their keys' dk and dv
 * sum the contributions of both responses.  Tensors, dtypes, streams,
 * status word and errors are as for swa_attn_fwd / swa_attn_bwd (which are
 * these calls with chosen_len = 0).  prompt_len >= 0, chosen_len >= 0 and
 * prompt_len + chosen_len <= L, else SWA_ERR_BAD_PLAN; a plan without a
 * chosen or without a rejected response is the plain causal window.  The
 * workspace sizes come from the *_prefix queries (pure host functions).
 */
size_t swa_attn_fwd_workspace_bytes_prefix(int B, int Hq, int Hkv, int L, int D, int window, int prompt_len,
                                            int chosen_len);
size_t swa_attn_bwd_workspace_bytes_prefix(int B, int Hq, int Hkv, int L, int D, int window, int prompt_len,
                                            int chosen_len);
int swa_attn_fwd_prefix(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, float* o, float* lse, int B,
                        int Hq, int Hkv, int L, int D, int window, int prompt_len, int chosen_len, float scale,
                        void* workspace, size_t workspace_bytes, void* stream);
int swa_attn_bwd_prefix(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o, const float* lse,
                        const swa_bf16* dO, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int L, int D,
                        int window, int prompt_len, int chosen_len, float scale, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * Attention sinks: swa_attn_fwd_ex / swa_attn_bwd_ex with one sink logit per
 * query head.  The pages name "sinks" only as a parameter of the attention
 * backward primitive, beside scale and causal ("Lab 028 lab detail: Off
 * NVIDIA, you fix the platform yourself", "What I changed, in plain terms"
 * item 2).  The reading taken is a per-head logit c_h that joins every row's
 * softmax normaliser and carries no value:
 *
 *   lse_i = ln( sum_{j in band(i)} exp(s_ij) + exp(c_h) )
 *   o_i   = sum_j exp(s_ij - lse_i) v_j
 *
 * and the backward also returns dc_h = - sum_{b, i} exp(c_h - lse_i) Delta_i
 * (Delta_i = dO_i . o_i), summed over the batch and the rows of head h.
 *
 *   sinks   [Hq] fp32, device memory, natural-log units (the units of
 *           scale * q . k); -inf is no sink.  Read only.  4-byte aligned.
 *   dsinks  [Hq] fp32, device memory, written (not accumulated).  4-byte
 *           aligned.
 *
 * q, k, v, o, lse, dO, dq, dk, dv, the geometry arguments, workspace
 * (sizes from swa_attn_*_workspace_bytes_ex), stream, status word and error
 * codes are as for swa_attn_fwd_ex / swa_attn_bwd_ex.  The backward reads the
 * lse the sink forward wrote; only dsinks needs the sinks themselves.  A
 * NULL sinks or dsinks is SWA_ERR_NULL_POINTER.  The decode path
 * (G * Lq <= 16) takes the sinks in its final normalisation too.
 */
int swa_attn_fwd_sinks(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* sinks, float* o,
                       float* lse, int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal, float scale,
                       void* workspace, size_t workspace_bytes, void* stream);
int swa_attn_bwd_sinks(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* sinks, const float* o,
                       const float* lse, const swa_bf16* dO, float* dq, float* dk, float* dv, float* dsinks, int B,
                       int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal, float scale, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Sequence sharding (context parallelism) with a halo: a sequence split into
 * contiguous chunks, one per rank, runs each chunk's queries over [halo;
 * own keys] through swa_attn_fwd_ex / swa_attn_bwd_ex (queries a suffix of
 * the keys).  The halo is the keys of earlier chunks that the chunk's
 * windows reach: the W - 1 keys before the chunk for a causal window W, all
 * earlier keys without a window.  This follows from the band structure
 * ("Lab 028 lab detail: Off NVIDIA, you fix the platform yourself", "What I
 * changed, in plain terms" items 3-4: a query only meets keys within the
 * window behind it); the pages do not describe the sharding itself.  The
 * backward of a chunk then holds dK / dV rows for halo keys that another rank
 * owns; that rank adds them into its own rows with this call:
 *
 *   dst[bh, row0 + r, d] += src[bh, r, d]   for bh < BH, r < nrows, d < D
 *
 * dst is [BH, dst_rows, D] fp32 (a rank's dk or dv, BH = B * Hkv), src is
 * [BH, nrows, D] fp32 (the halo rows received); device pointers, 16-byte
 * aligned, D a multiple of 4, 0 <= row0 and row0 + nrows <= dst_rows.
 * Asynchronous on `stream`.  Returns SWA_OK, SWA_ERR_NULL_POINTER,
 * SWA_ERR_BAD_SHAPE, SWA_ERR_MISALIGNED or SWA_ERR_CUDA.
 */
int swa_attn_add_rows_f32(float* dst, const float* src, int BH, int dst_rows, int row0, int nrows, int D,
                          void* stream);

/*
 * Forward.  Reads q [B,Hq,L,D], k and v [B,Hkv,L,D] (bf16); writes
 * o [B,Hq,L,D] (fp32, normalised attention output) and lse [B,Hq,L] (fp32,
 * natural-log sum over the band of exp(scale * q_i . k_j)).  The forward
 * writes the logsumexp the backward reuses ("Lab 028 lab detail", "What I
 * changed, in plain terms" item 1).
 * Returns SWA_OK or a negative SWA_ERR_* code; on an argument error nothing
 * is enqueued.
 */
int swa_attn_fwd(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, float* o, float* lse,
                 int B, int Hq, int Hkv, int L, int D, int window, float scale,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Workspace bytes swa_attn_bwd needs for this shape: O(B*Hq*L) floats for
 * the row term Delta plus any per-call operand staging.  Pure host function.
 */
size_t swa_attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int L, int D, int window);

/*
 * Backward of o with respect to q, k, v given the upstream gradient dO.
 * Reads q, k, v, dO (bf16), o and lse (fp32, from swa_attn_fwd with the same
 * arguments); writes dq [B,Hq,L,D], dk and dv [B,Hkv,L,D] (fp32).
 * Recomputes P from lse instead of storing it ("Training -- design",
 * section 6: store per-row LSE, recompute P), computes
 * Delta_i = dO_i . o_i, dS = P (dP - Delta), and visits only key/query tile
 * pairs that intersect the band ("Lab 028 lab detail", "What I changed, in
 * plain terms" item 3).  dk and dv sum over the Hq/Hkv query heads of each
 * kv head.  Deterministic: no floating-point atomics.
 * Returns SWA_OK or a negative SWA_ERR_* code; on an argument error nothing
 * is enqueued.
 */
int swa_attn_bwd(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o,
                 const float* lse, const swa_bf16* dO, float* dq, float* dk, float* dv,
                 int B, int Hq, int Hkv, int L, int D, int window, float scale,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Device-side status of the current device: synchronises `stream`, returns
 * the first SWA_ERR_* code latched by a kernel since the previous call (or
 * SWA_OK), and clears it.  Returns SWA_ERR_CUDA if the CUDA calls fail.
 */
int swa_attn_get_status(void* stream);

/*
 * swa_attn_selftest_timeout: exercises the device-side failure path without
 * a fault.  It launches, on `stream`, one CTA that waits on a barrier that
 * nothing completes.  The wait uses the same bounded wait as every kernel of
 * the library, with a limit of about 1 ms.  When that limit runs out, the CTA
 * latches SWA_ERR_DEVICE_TIMEOUT in the status word, and the next
 * swa_attn_get_status() on the stream returns it.  The CUDA context stays
 * usable.  Returns SWA_OK, or SWA_ERR_CUDA if the launch fails.
 */
int swa_attn_selftest_timeout(void* stream);

/* Static, human-readable description of a return code. */
const char* swa_attn_strerror(int code);

/*
 * swa_attn_bwd_noalloc: the backward of swa_attn_bwd, for callers that
 * cannot allocate device memory or pass a workspace -- for example code whose
 * device memory all belongs to a host framework's allocator, or a plugin
 * entry point whose fixed signature has no workspace argument.  (The pages
 * have no counterpart; this is a deployment convenience of this library.)
 *
 * It computes the same quantities but runs fp32 kernels on the CUDA cores,
 * not the tensor cores: no fp16 operand copies (any finite bf16 input is
 * exact), and a throughput bound of about 80 TFLOP/s (152 SMs x 128 fp32
 * lanes x 2 flop x 2.07 GHz) against roughly a petaflop for swa_attn_bwd on
 * the same shapes.  Its results match swa_attn_bwd within the parity
 * tolerance of this library, not bit for bit.
 *
 * It takes no workspace: the per-row term Delta lives in a fixed array built
 * into the library (8 MiB of fp32 on every GPU that loads the library, held
 * until the process exits), so it supports B * Hq * L <= 2,097,152 and
 * returns SWA_ERR_NOALLOC_LIMIT above that.  It calls no cudaMalloc or
 * cudaFree.  Its first call on a device looks up that array's device address
 * (cudaGetSymbolAddress, with the device current); make that first call
 * before any stream capture begins.  Every call shares the one array: calls
 * whose kernels overlap on the GPU race on it, so serialise them (one stream,
 * or events).  Other arguments, layouts, outputs and errors are as for
 * swa_attn_bwd.
 */
int swa_attn_bwd_noalloc(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o,
                         const float* lse, const swa_bf16* dO, float* dq, float* dk, float* dv,
                         int B, int Hq, int Hkv, int L, int D, int window, float scale,
                         void* stream);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int swa_attn_version(void);

/*
 * Optional kernel timing, for benchmarks.  Between swa_attn_profile_begin()
 * and swa_attn_profile_end(), every kernel this library launches (from any
 * host thread, on any stream of any device) is bracketed by two CUDA events
 * recorded on the launch stream.  profile_end() waits for those events and
 * writes per-kernel totals into out[0 .. *n_out - 1] (at most max_entries;
 * kernels are named by what they compute).  This mode allocates host memory
 * and CUDA events per launch; it is the only one that allocates host memory.
 */
typedef struct {
    char name[48];       /* kernel name, NUL-terminated */
    long long launches;  /* launches recorded */
    double total_ms;     /* summed event-measured duration */
} swa_attn_kernel_time;

int swa_attn_profile_begin(void);
int swa_attn_profile_end(swa_attn_kernel_time* out, int max_entries, int* n_out);

#ifdef __cplusplus
}
#endif

#endif /* SWA_ATTN_H */
