/*
 * la.h -- C ABI of the GB300 (sm_103a) causal linear attention library (libla).
 *
 * The library computes attention with the kernel feature map phi(x) = elu(x) + 1
 * (alpha = 1):
 *
 *   o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i),
 *   S_i = sum_{j in J(i)} phi(k_j) v_j^T   (Dk x Dv),   z_i = sum_{j in J(i)} phi(k_j)   (Dk),
 *
 * with J(i) = {j <= i} for the causal forms and all j for the non-causal form.
 * No 1/sqrt(D) scale and no epsilon are applied.
 *
 * Sources, by page title and section:
 *   "Transformers은 RNN이다 — 선형 어텐션으로 빠른 Autoregressive Transformer
 *    만들기" (irregular6612 digest): Methods; 핵심 구성요소 1-4.
 *   "[논문 리뷰] Transformers are RNNs: Fast Autoregressive Transformers with
 *    Linear Attention" (velog review): 3.2 Linearized Attention, 3.3 Feature
 *    Maps, 3.4 Causal Masking, 3.5 Gradient Computation, 3.6 Transformers and RNNs.
 *   "선형 어텐션" (itwiki): 결합 법칙으로 순서 바꾸기; 인과 마스킹과 순환형;
 *    계산 형태 비교 (chunked form); 구현.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * Layout.   q, k: [B, H, N, Dk]; v, o, dout: [B, H, N, Dv]; dense row-major
 *           (innermost dimension contiguous), one dtype per call (la_shape.dtype).
 *           Decode state S: [B, H, Dk, Dv] fp32; z: [B, H, Dk] fp32.
 * Memory.   Every tensor pointer is a DEVICE pointer on the current CUDA device,
 *           16-byte aligned.  The caller owns and allocates every buffer,
 *           including the workspace; the library allocates no device memory and
 *           keeps no per-call state.  The workspace is scratch for one call: its
 *           contents on entry are ignored and on exit are unspecified.
 * Sizes.    B, H, N >= 0 (any zero makes the call a no-op returning LA_OK; the
 *           pointers may then be NULL).  Dk and Dv are each one of 16, 32, 64,
 *           128.  B*H <= 65535 and B*H*N*max(Dk,Dv) < 2^40.
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *           work is enqueued asynchronously on it; the call returns once the
 *           launches are queued.
 * Errors.   Invalid arguments return LA_ERR_INVALID_ARG, unsupported sizes
 *           LA_ERR_UNSUPPORTED and a short workspace LA_ERR_WORKSPACE, all before
 *           anything is launched.  A failed launch returns LA_ERR_CUDA.  Faults
 *           detected on the device (a bounded wait that ran out) are recorded in
 *           a sticky device word that la_last_error() reads after the stream has
 *           been synchronised.  No C++ exception crosses this interface.
 * Precision. Accumulation is fp32 throughout; inputs and outputs are fp32 or
 *           bf16 (la_shape.dtype); the decode state is always fp32.
 */
#ifndef LA_H_
#define LA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, negative size, bad dtype or op */
    LA_ERR_UNSUPPORTED = 2,  /* Dk or Dv not in {16, 32, 64, 128}, B*H > 65535, or not an sm_103 device */
    LA_ERR_WORKSPACE = 3,    /* ws_bytes smaller than la_workspace_bytes(), or ws NULL */
    LA_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    LA_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out (read via la_last_error) */
    LA_ERR_BOUNDS = 6        /* debug builds only: a device-side index check failed and the access
                                was skipped (read via la_last_error; la_error_detail names the site) */
} la_status;

typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

typedef enum {
    LA_OP_NONCAUSAL_FWD = 0,
    LA_OP_CAUSAL_FWD = 1,
    LA_OP_CAUSAL_BWD = 2,
    LA_OP_NONCAUSAL_BWD = 3,
    LA_OP_RETENTION_FWD = 4
} la_op;

/* Problem shape.  dtype is an la_dtype value. */
typedef struct {
    int B, H, N, Dk, Dv;
    int dtype;
} la_shape;

/* A cudaStream_t, declared opaquely so this header needs no CUDA headers. */
typedef struct CUstream_st* la_stream_t;

/*
 * Workspace bytes the call `op` needs for shape `s` (0 when none).  A pure
 * function of (op, s): it does not touch the device.  Returns 0 for invalid
 * arguments as well; the call itself then reports the error.
 */
size_t la_workspace_bytes(int op, la_shape s);

/*
 * Non-causal linear attention, o_i = phi(q_i)^T S / phi(q_i)^T z with
 * S = phi(K)^T V and z = phi(K)^T 1 summed over all N positions of the head.
 * ("Transformers은 RNN이다" digest, 핵심 구성요소 2; velog review 3.2;
 * itwiki 결합 법칙으로 순서 바꾸기.)
 * q, k: [B,H,N,Dk]; v: [B,H,N,Dv]; o: [B,H,N,Dv] (written).
 */
la_status la_noncausal_fwd(const void* q, const void* k, const void* v, void* o, la_shape s,
                           void* ws, size_t ws_bytes, la_stream_t stream);

/*
 * Causal linear attention (j <= i, diagonal included), computed in the chunked
 * form: inside a chunk the masked product phi(Q_c) phi(K_c)^T is formed, and the
 * state (S, z) is carried between chunks by a prefix sum.  A final chunk shorter
 * than the chunk size is masked.  (Digest, 핵심 구성요소 3; velog review 3.4;
 * itwiki 계산 형태 비교, chunked row, and 구현.)
 * q, k: [B,H,N,Dk]; v: [B,H,N,Dv]; o: [B,H,N,Dv] (written).
 * Runs as three launches: the segments' own sums, their exclusive scan and the
 * output pass.  The workspace keeps every segment's starting state for
 * la_causal_bwd_after_fwd.
 */
la_status la_causal_fwd(const void* q, const void* k, const void* v, void* o, la_shape s,
                        void* ws, size_t ws_bytes, la_stream_t stream);

/*
 * la_causal_fwd as one kernel launch (after a memset of a few KB of flags in the
 * workspace) for bf16 heads of 64 or 128; other shapes run la_causal_fwd.
 * Arguments, workspace and results are those of la_causal_fwd, bit for bit: each
 * block forms its segment's own sums, publishes them, adds the earlier segments'
 * (a chained scan in segment order, the separate scan's additions exactly) and
 * writes the outputs.  Every wait is bounded: one that runs out records
 * LA_ERR_TIMEOUT in the sticky word and the block ends.  Blocks take their work
 * from a ticket counter, so a block only waits on blocks already running.  It
 * saves two launches; it is not faster at the sizes measured, because a block
 * adds the earlier segments' published sums one L2 round trip at a time while
 * their prefixes are not yet complete.
 */
la_status la_causal_fwd_fused(const void* q, const void* k, const void* v, void* o, la_shape s,
                              void* ws, size_t ws_bytes, la_stream_t stream);

/*
 * la_causal_fwd that also returns the state after the last position, the (S, z)
 * from which la_recurrent_step continues the sequence (prefill, then one step
 * per new token: the RNN view of the causal form, digest 핵심 구성요소 4 and
 * velog review 3.6):  S = phi(K)^T V  [B,H,Dk,Dv] and  z = phi(K)^T 1  [B,H,Dk],
 * summed over all N positions of each head, fp32, written (not accumulated).
 * For N = 0 both are set to zero.  o and the workspace as for la_causal_fwd.
 * Costs one more pass over k and v of the last segment of each head.
 */
la_status la_causal_fwd_with_state(const void* q, const void* k, const void* v, void* o,
                                   float* S, float* z, la_shape s,
                                   void* ws, size_t ws_bytes, la_stream_t stream);

/*
 * Gradient of the causal form for an upstream gradient dout = dL/do.  States
 * are recomputed from q, k, v (nothing from the forward call is needed), and
 * no per-position state is stored, so memory stays linear in N ("velog review"
 * 3.5 Gradient Computation: the gradient is itself a cumulative sum).  With
 * den_i = phi(q_i)^T z_i, P_i = dout_i / den_i, g_i = -(dout_i . o_i) / den_i,
 * R_j = sum_{i>=j} phi(q_i) P_i^T and r_j = sum_{i>=j} g_i phi(q_i):
 *   dq_i = (S_i P_i + g_i z_i) * phi'(q_i),
 *   dk_j = (R_j v_j + r_j) * phi'(k_j),
 *   dv_j = R_j^T phi(k_j).
 * q, k, dq, dk: [B,H,N,Dk]; v, dout, dv: [B,H,N,Dv]; dq, dk, dv written.
 */
la_status la_causal_bwd(const void* q, const void* k, const void* v, const void* dout,
                        void* dq, void* dk, void* dv, la_shape s,
                        void* ws, size_t ws_bytes, la_stream_t stream);

/*
 * The same gradient as la_causal_bwd, bit for bit, for the training step in
 * which the forward has just run: the forward state entering each segment is
 * taken from the workspace of that la_causal_fwd call instead of being summed
 * again from k and v.  This keeps the memory bound of the cumulative-sum
 * gradient (velog review 3.5): what is kept from the forward is one state per
 * segment, not one per position.
 * fwd_ws: the workspace (at least la_workspace_bytes(LA_OP_CAUSAL_FWD, s)
 * bytes) of an la_causal_fwd call on the same q, k, v and shape, unchanged
 * since and complete in stream order; it is read, not written.  ws: a
 * backward workspace as for la_causal_bwd.  A forward workspace that is too
 * small returns LA_ERR_WORKSPACE; one from another shape or other inputs gives
 * wrong gradients (this is not detectable).
 */
la_status la_causal_bwd_after_fwd(const void* q, const void* k, const void* v, const void* dout,
                                  void* dq, void* dk, void* dv, la_shape s,
                                  const void* fwd_ws, size_t fwd_ws_bytes,
                                  void* ws, size_t ws_bytes, la_stream_t stream);

/*
 * Gradient of the non-causal form (la_noncausal_fwd) for an upstream gradient
 * dout.  With S = phi(K)^T V and z = phi(K)^T 1 over all positions,
 * den_i = phi(q_i)^T z, P_i = dout_i / den_i, g_i = -(dout_i . o_i) / den_i,
 * R = sum_i phi(q_i) P_i^T and r = sum_i g_i phi(q_i) (all i):
 *   dq_i = (S P_i + g_i z) * phi'(q_i),  dk_j = (R v_j + r) * phi'(k_j),  dv_j = R^T phi(k_j).
 * (The same state algebra as the causal gradient without the mask: velog
 * review 3.2 and 3.5; digest 핵심 구성요소 2.)  A query pass computes dq and the
 * sums of R and r, a key pass dk and dv; the pages print no formula for this
 * gradient, it is derived from the definition by the chain rule.
 * Shapes as for la_causal_bwd; workspace la_workspace_bytes(LA_OP_NONCAUSAL_BWD, s).
 */
la_status la_noncausal_bwd(const void* q, const void* k, const void* v, const void* dout,
                           void* dq, void* dk, void* dv, la_shape s,
                           void* ws, size_t ws_bytes, la_stream_t stream);

/*
 * One training step of the causal form on host-resident data: o = the causal
 * forward of (q, k, v), then (dq, dk, dv) = its gradient for dout, exactly as
 * la_causal_fwd followed by la_causal_bwd_after_fwd on each group of heads.
 * All eight tensors are pinned (page-locked) host buffers in the [B,H,N,D]
 * layout of the device calls.  Heads are independent, so the call cuts the B*H
 * heads into groups of `group_heads` consecutive heads and overlaps, on three
 * internal streams, the host->device copies of one group, the kernels of the
 * previous one and the device->host copies of the one before; the transfers,
 * not the kernels, then bound the step.  dev_buf: device scratch of at least
 * la_host_step_bytes(s, group_heads) bytes, owned by the caller (two slots of
 * group buffers and the two workspaces).  The work starts after what is
 * already queued on `stream`, and `stream` waits for all of it: read the
 * outputs after synchronising it.  Concurrent calls on one device share the
 * internal streams and must not overlap.  Pageable host memory is refused
 * (LA_ERR_INVALID_ARG).  The internal streams and events are created on the
 * first call on a device and kept.
 */
size_t la_host_step_bytes(la_shape s, int group_heads);
la_status la_causal_step_host(const void* q, const void* k, const void* v, const void* dout,
                              void* o, void* dq, void* dk, void* dv, la_shape s,
                              int group_heads, void* dev_buf, size_t dev_bytes, la_stream_t stream);

/*
 * One recurrent (decode) step for every head, the state updated first and then
 * read:  S <- S + phi(k) v^T,  z <- z + phi(k),  out = phi(q)^T S / phi(q)^T z.
 * ("Transformers은 RNN이다" digest, 핵심 구성요소 4; velog review 3.6; itwiki
 * 인과 마스킹과 순환형.)
 * q, k: [B,H,Dk]; v, out: [B,H,Dv] in s.dtype; S: [B,H,Dk,Dv] fp32 and
 * z: [B,H,Dk] fp32, both read and updated in place.  s.N is ignored.  The
 * caller zeroes S and z before the first step of a sequence; passing saved
 * (S, z) back in resumes it exactly.  No workspace.
 */
la_status la_recurrent_step(const void* q, const void* k, const void* v, float* S, float* z,
                            void* out, la_shape s, la_stream_t stream);

/*
 * Retention: causal linear attention with a constant decay per head, the
 * decayed update of itwiki 선형 어텐션, section 발전: 감쇠, 게이트, 델타 규칙
 * (RetNet's gamma):
 *   S_t = gamma_h S_(t-1) + k_t v_t^T  (S_(-1) = 0),   o_t = S_t^T q_t,
 * i.e. o_t = sum_(j<=t) gamma_h^(t-j) (q_t . k_j) v_j.  The feature map is the
 * identity and there is no normaliser (phi and z above do not enter), so
 * gamma = 1 gives the plain masked product tril(Q K^T) V, and gamma = 0 gives
 * o_t = (q_t . k_t) v_t (0^0 = 1).  Computed in the chunked form: a decay mask
 * gamma^(a-b) inside a chunk of C = 64 positions, the carried state seen
 * through gamma^(a+1), and a decayed prefix scan over segments of chunks.
 * q, k: [B,H,N,Dk]; v, o: [B,H,N,Dv] in s.dtype; o written.
 * gamma: DEVICE pointer to H fp32 values (one per head, shared by the B batch
 *   entries), 4-byte aligned, read only.  Any real value is computed as
 *   written; the method intends 0 <= gamma <= 1 (|gamma| > 1 grows without
 *   bound).
 * S: NULL, or a DEVICE fp32 [B,H,Dk,Dv] that receives the state after the
 *   last position (written, not accumulated; zero for N = 0), from which
 *   la_retention_step continues the sequence.
 * Workspace: la_workspace_bytes(LA_OP_RETENTION_FWD, s).
 */
la_status la_retention_fwd(const void* q, const void* k, const void* v, const float* gamma,
                           void* o, float* S, la_shape s,
                           void* ws, size_t ws_bytes, la_stream_t stream);

/*
 * One decode step of retention for every head, the state updated first and
 * then read:  S <- gamma_h S + k v^T,  out = S^T q.
 * q, k: [B,H,Dk]; v, out: [B,H,Dv] in s.dtype; gamma as for la_retention_fwd;
 * S: [B,H,Dk,Dv] fp32, read and updated in place (zero before the first step
 * of a sequence, or the S of la_retention_fwd).  s.N is ignored.  No workspace.
 */
la_status la_retention_step(const void* q, const void* k, const void* v, const float* gamma,
                            float* S, void* out, la_shape s, la_stream_t stream);

/*
 * la_causal_fwd with no workspace argument: the same causal forward, with its
 * scratch (the per-segment states) in a 16 MiB device array that the library
 * owns.  The pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory when they call the library, such as a
 * plugin inside a host framework that owns every device allocation and hands
 * its plugins no workspace, or a latency-critical loop that may not call
 * cudaMalloc (which can synchronise the device) after start-up.
 * Arguments, layouts, dtypes and checks are those of la_causal_fwd.  It calls
 * no cudaMalloc, cudaFree or other allocating routine.  The array is static:
 * every GPU that loads the library holds the 16 MiB until the process exits.
 * The first call on a device looks up the array's address on that device
 * (that device must be current) and caches it with the current CUDA context;
 * a call under another context of the device (after cudaDeviceReset, say)
 * looks it up again.  Make the first call on a device, and the first after a
 * reset, before any stream capture.  The array holds one state record per
 * head and segment, and needs room for at least one segment: B*H records of
 * (Dk*Dv + Dk)*4 bytes on the CUDA-core path, and of (128*128 + 128)*4 bytes
 * on the tensor-core path (bf16 heads of 64 or 128 keep the padded 128-wide
 * record), so B*H may be at most 254 for bf16 heads of 64 or 128.  Larger
 * sizes return LA_ERR_WORKSPACE before anything is launched; where the usual
 * segment count does not fit, fewer, longer segments are used.  Every call shares the array, so calls whose work
 * overlaps on the GPU (other streams or host threads) race on it and corrupt
 * each other's results: serialise them.  Each call rewrites every part of the
 * array it reads, so what a previous call left there does not matter.
 */
la_status la_causal_fwd_noalloc(const void* q, const void* k, const void* v, void* o, la_shape s,
                                la_stream_t stream);

/*
 * Sticky device-side status: LA_OK, or the first error a kernel recorded since
 * the last la_clear_error() (LA_ERR_TIMEOUT for a bounded wait that ran out;
 * LA_ERR_BOUNDS for a failed index check of the debug build, whose source file
 * and line la_error_detail() then gives).
 * It reads device memory synchronously (the current device is synchronised);
 * call it after the stream work has finished.  la_clear_error() resets it.
 */
la_status la_last_error(void);
la_status la_clear_error(void);

/*
 * Self-test of the device-side failure detection, with no fault: launches one
 * thread that waits on an mbarrier phase nothing completes.  Like every wait in
 * the library's kernels, the wait is bounded (about one second of SM clock);
 * it gives up, records LA_ERR_TIMEOUT in the sticky status word and the kernel
 * ends normally.  After the stream has been synchronised, la_last_error()
 * returns LA_ERR_TIMEOUT (unless an earlier error is already recorded); clear it
 * with la_clear_error().  The device and context stay usable.
 */
la_status la_selftest_bounded_wait(la_stream_t stream);

/*
 * Self-test of the one-launch causal forward's chained scan, with no fault:
 * la_causal_fwd on the given buffers (same arguments and checks), except that
 * the block of segment 0 of head 0 never publishes its sums.  The later blocks
 * of that head wait for it; each wait gives up after about one second, records
 * LA_ERR_TIMEOUT in the sticky status word and the block ends; all other heads
 * complete normally.  Needs a shape that runs the one-launch forward with at
 * least two segments per head (bf16, Dk = Dv = 64 or 128), else returns
 * LA_ERR_INVALID_ARG before anything is launched.  o (head 0) and the workspace
 * are left unspecified.  The device and context stay usable.
 */
la_status la_selftest_lookback_timeout(const void* q, const void* k, const void* v, void* o, la_shape s,
                                       void* ws, size_t ws_bytes, la_stream_t stream);

/* Static description of a status code. */
const char* la_status_string(la_status st);

/* Text of the most recent host-side failure on the calling thread ("" if none). */
const char* la_error_detail(void);

/*
 * Library version, e.g. "0.1.1".  A build with device-side bounds checks (the
 * debug build: every plain global-memory access, segment record, TMA tile
 * coordinate and shared-memory tile offset of the kernels is checked against
 * the extents of its tensor, and a failed check records LA_ERR_BOUNDS and skips
 * the access instead of trapping) reports "<version>-debug".
 */
const char* la_version(void);

/*
 * Per-kernel timing (for the benchmark).  While enabled, every kernel launch
 * is bracketed by CUDA events recorded on its launch stream; la_timing_read()
 * synchronises those events and reports, per kernel name, the number of
 * launches and their total device time since the last reset.  Off by default;
 * enabling it adds two event records per launch and nothing else.
 */
typedef struct {
    const char* name;   /* static string owned by the library */
    int launches;
    double total_ms;
} la_kernel_time;

la_status la_timing_enable(int on);
la_status la_timing_reset(void);
/* Fills up to `max` entries; returns the number of distinct kernels, or -1 on error. */
int la_timing_read(la_kernel_time* out, int max);

#ifdef __cplusplus
}
#endif

#endif /* LA_H_ */
