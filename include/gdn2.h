/*
 * gdn2.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet-2 chunked prefill
 * forward.
 *
 * The operation is the GDN-2 recurrence of the FlashInfer docs page
 * "flashinfer.gdn2_prefill.chunk_gated_delta_rule2" (op description), per
 * sequence n and state head hs (see gdn2_dims for the head counts):
 *
 *     S_t   = diag(exp(g_t)) S_{t-1}
 *     u_t   = w_t * v_t - (beta_t * k_t)^T S_t
 *     S_t  += k_t u_t^T
 *     o_t   = scale * q_t^T S_t
 *
 * S is a K x V fp32 matrix.  The library evaluates it in 64-token chunks in
 * WY form (FlashRT gated-delta-attention page, "64-token WY blocks"; burn-gdn2
 * README, "Fused CUDA kernels" and "Numerical stability") over packed
 * variable-length sequences, as the FlashInfer docs' argument list describes.
 *
 * Conventions common to every entry point:
 *  - All tensor pointers are DEVICE pointers unless stated otherwise.
 *  - The caller owns every buffer, the workspace included.  The library never
 *    allocates device memory, never synchronises the stream (except
 *    gdn2_device_status, which says so) and never writes its inputs.
 *  - Functions return a gdn2_status; GDN2_OK is 0.  Argument errors are found
 *    on the host before anything is enqueued, so a non-zero return from
 *    argument checking means nothing was launched.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All work is enqueued asynchronously on it.
 *  - The library is built for sm_103a only; other devices get GDN2_ERR_ARCH.
 */
#ifndef GDN2_H
#define GDN2_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN2_API __attribute__((visibility("default")))
#else
#define GDN2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn2_status {
    GDN2_OK = 0,
    GDN2_ERR_NULL = 1,        /* a required pointer is NULL                          */
    GDN2_ERR_SHAPE = 2,       /* unsupported sizes (K, V), HV % H != 0, N < 0, ...    */
    GDN2_ERR_STRIDE = 3,      /* innermost stride != 1, or a stride / base pointer    */
                              /* is not a multiple of 16 bytes                        */
    GDN2_ERR_ALIAS = 4,       /* out or final_state overlaps an input                 */
    GDN2_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than gdn2_workspace_bytes  */
    GDN2_ERR_ARCH = 6,        /* current device is not compute capability 10.3        */
    GDN2_ERR_LAUNCH = 7,      /* a kernel launch failed (cudaGetLastError)            */
    GDN2_ERR_DTYPE = 8,       /* unsupported dtype code                               */
    GDN2_ERR_CU_SEQLENS = 9,  /* device-side: cu_seqlens[0] != 0, decreasing, or      */
                              /* cu_seqlens[N] != T_tot (see gdn2_device_status)      */
    GDN2_ERR_CUDA = 10,       /* another CUDA runtime error                           */
    GDN2_ERR_IMPL = 11,       /* unknown implementation selector                      */
    GDN2_ERR_TIMEOUT = 12,    /* device-side: a kernel gave up waiting on one of its  */
                              /* own pipeline barriers (see gdn2_device_status)       */
    GDN2_ERR_NOALLOC_LIMIT = 13, /* the problem needs more scratch than               */
                              /* gdn2_chunk_fwd_noalloc holds                         */
    GDN2_ERR_RANGE = 14,      /* device-side: a value passed the range of the fp16    */
                              /* intermediates and was clipped; outputs are invalid   */
                              /* (see gdn2_device_status)                             */
    GDN2_ERR_BOUNDS = 15      /* device-side, checked builds only (compiled with      */
                              /* GDN2_CHECK_BOUNDS): an index left its buffer; a      */
                              /* library defect, outputs invalid                      */
} gdn2_status;

typedef enum gdn2_dtype {
    GDN2_DTYPE_BF16 = 0,
    GDN2_DTYPE_F16 = 1,
    GDN2_DTYPE_F32 = 2
} gdn2_dtype;

typedef enum gdn2_impl {
    GDN2_IMPL_TC = 0,    /* default: tcgen05 / TMA kernels                          */
    GDN2_IMPL_SIMT = 1   /* CUDA-core fp32 kernels of the same chunked algorithm;    */
                         /* a second GPU path for cross-checks, never a fallback     */
} gdn2_impl;

/*
 * Problem description.  Every token-major tensor X has element strides
 * x_stride[0] (between tokens) and x_stride[1] (between heads); its innermost
 * (channel) stride is 1 (FlashInfer docs: "only the innermost dimension has
 * to be contiguous").  Strides are in ELEMENTS of that tensor's dtype and,
 * like base pointers, must be multiples of 16 bytes.
 *
 * Heads (FlashInfer docs, parameters q, k, v): H query heads, HK key heads
 * (HK = 0 means H) and HV value heads, where HK equals H or HV and H, HV are
 * equal or one a multiple of the other.  There is one state per STATE head
 * hs < HS = max(H, HV) (the docs' num_sab_heads; also the output heads);
 * state head hs reads query head hs / (HS / H), key head hs / (HS / HK) and
 * value head hs / (HS / HV), contiguous groups of state heads sharing one.
 *
 *   q             [T_tot, H,  K]   dtype_qkv (bf16 or fp16)
 *   k             [T_tot, HK, K]   dtype_qkv
 *   v             [T_tot, HV, V]   dtype_qkv
 *   w             [T_tot, HS, V]   dtype_qkv (write gate)
 *   g             [T_tot, HS, K]   dtype_g: fp32, bf16 or fp16 (natural-log decay, <= 0)
 *   beta          [T_tot, HS, K]   dtype_qkv (erase gate, post-sigmoid; [0, 2] allowed)
 *   out           [T_tot, HS, V]   dtype_qkv
 *   initial_state [N, HS, K, V]    dtype_state (fp32 or bf16), contiguous, K-major
 *                                  (row c = key channel); [N, HS, V, K] when
 *                                  state_v_major = 1 (the FlashInfer docs' layout)
 *   final_state   same dtype and layout as initial_state
 *   cu_seqlens    [N + 1]          int32 (or int64 with cu_seqlens_i64 = 1)
 *
 * (FlashInfer docs, chunk_gated_delta_rule2 parameters: q/k/v fp16 or bf16,
 * beta and w read at q's dtype, g fp32/bf16/fp16, state fp32 or bf16.)  The
 * SIMT implementation supports only the defaults (bf16, fp32 g, fp32 K-major
 * state); other combinations with impl = GDN2_IMPL_SIMT are GDN2_ERR_DTYPE.
 *
 * Supported sizes: K = V in {64, 128}; the head counts above; N >= 0;
 * T_tot >= 0 (T_tot = 0 writes only final_state = initial_state).
 */
typedef struct gdn2_dims {
    int64_t T_tot;
    int32_t N, H, HV, K, V;
    int64_t q_stride[2], k_stride[2], v_stride[2], g_stride[2];
    int64_t beta_stride[2], w_stride[2], o_stride[2];
    int32_t dtype_qkv;      /* GDN2_DTYPE_BF16 or GDN2_DTYPE_F16 (q, k, v, beta, w, out) */
    int32_t dtype_g;        /* GDN2_DTYPE_F32, GDN2_DTYPE_BF16 or GDN2_DTYPE_F16  */
    int32_t cu_seqlens_i64; /* 0: int32 cu_seqlens, 1: int64                      */
    int32_t use_qk_l2norm;  /* 1: divide q, k rows by max(||x||_2, 1e-12) first   */
                            /* (FlashInfer docs: use_qk_l2norm_in_kernel)         */
    int32_t impl;           /* gdn2_impl                                          */
    int32_t state_v_major;  /* 0: states [N, HS, K, V]; 1: [N, HS, V, K]          */
    int32_t dtype_state;    /* GDN2_DTYPE_F32 or GDN2_DTYPE_BF16                  */
    int32_t state_segments; /* chunk-parallel state pass; see below               */
    int32_t HK;             /* key heads; 0 = H (the query heads)                 */
} gdn2_dims;
/*
 * state_segments (tensor-core path, K = V = 128): P > 1 splits each
 * sequence's chunks into P segments of ceil(chunks / P).  Every segment's
 * state map is affine, S_out = M S_in + B.  The library replays segment 0
 * from the initial state while it computes [M | B] for segments 1 .. P - 2
 * in parallel, combines those in order into each later segment's incoming
 * state (fp32 accumulation of products whose operands are split into bf16
 * high and low parts, about 16 mantissa bits each), then replays segments
 * 1 .. P - 1 in parallel for o and the final state.  This shortens the
 * sequential chain for few (sequence, head) pairs on long sequences (the
 * FlashInfer docs, output_state: the cuDNN engine splits one sequence
 * across CTAs).  0 = the library chooses
 * P from a time model of the passes (P > 1 only for few (sequence, head)
 * pairs on long sequences), 1 = one sequential pass, 2 .. 64 forced.
 * Out of range, or > 1 with the SIMT path or K != 128: GDN2_ERR_SHAPE.  M is
 * formed with the same 16-bit operands as the state pass, so results differ
 * from the sequential pass by rounding only.  gdn2_recurrent_fwd checks only
 * the range.
 */

/*
 * Bytes of device workspace gdn2_chunk_fwd needs for `dims` (0 if dims is
 * NULL or invalid).  The workspace holds the device-built chunk map, a status
 * word and the chunk intermediates; it may be reused across calls that do
 * not overlap on the GPU.  Host-only; no CUDA call.
 */
GDN2_API size_t gdn2_workspace_bytes(const gdn2_dims *dims);

/*
 * Fill `dims` for contiguous tensors of the given sizes (strides = packed
 * row-major), key heads = query heads (HK = 0), dtype_qkv = bf16, dtype_g =
 * fp32, int32 cu_seqlens, no L2 norm, impl = GDN2_IMPL_TC, fp32 K-major
 * states.  H is the query (and key) head count, HV the value head count.
 * Host-only.
 */
GDN2_API gdn2_status gdn2_dims_init(gdn2_dims *dims, int64_t T_tot, int32_t N, int32_t H, int32_t HV,
                           int32_t K, int32_t V);

/*
 * Validate arguments exactly as gdn2_chunk_fwd does, without touching the
 * device: pointers, sizes, strides, dtypes, aliasing and workspace size.
 * Host-only; returns the status gdn2_chunk_fwd would return before launching.
 */
GDN2_API gdn2_status gdn2_check_args(const void *q, const void *k, const void *v, const void *g,
                            const void *beta, const void *w, const void *initial_state,
                            const void *cu_seqlens, const void *out, const void *final_state,
                            const gdn2_dims *dims, const void *workspace,
                            size_t workspace_bytes);

/*
 * The chunked GDN-2 prefill forward (FlashInfer docs, chunk_gated_delta_rule2:
 * signature and parameters; the argument order follows it).
 *
 *   g             may be NULL: no decay (g = 0)
 *   beta          may be NULL: beta = 1
 *   w             may be NULL: w = 1
 *   scale         query scale; <= 0 means 1/sqrt(K)
 *   initial_state may be NULL: zero state
 *   final_state   may be NULL: not written.  Must not overlap initial_state.
 *   out           written in place; must not overlap any input
 *   workspace     device buffer of at least gdn2_workspace_bytes(dims) bytes
 *
 * Chunks are 64 tokens and never span two sequences; an empty sequence
 * returns final_state = initial_state.  Numerics: bf16 tensor-core operands
 * for the decayed q.k and k.k products, fp16 operands for the chunk
 * intermediates, fp32 accumulation and fp32 carried state.  Chunk-local decays
 * are applied through 16-token sub-chunk references (burn-gdn2 README,
 * "Numerical stability"): every factor across sub-chunks is <= 1, and inside
 * a sub-chunk a key channel that decays by more than 2^92 (63.8 nats) takes
 * its decay per token pair exactly, so any g <= 0 is valid.  Values of the
 * fp16 intermediates (which scale with v, w and the state) must stay below
 * 65504 in magnitude: a value past that is clipped and the call reports
 * GDN2_ERR_RANGE through gdn2_device_status (outputs then invalid).
 *
 * Returns GDN2_OK once all kernels are enqueued.  cu_seqlens is checked on
 * the device; a bad cu_seqlens makes every kernel a no-op and is reported by
 * gdn2_device_status.
 *
 * The tensor-core path reads g, v and w through TMA tensor maps encoded on
 * the host at each call (no device state).  Where the driver rejects a layout
 * (for example a zero head stride) it copies those rows one by one instead;
 * the environment variable GDN2_ROW_COPIES=1 forces that path (diagnostics).
 * The sequential state pass runs kernels with a one-chunk lookahead (one for
 * 64-column V tiles, used when few (sequence, head) pairs leave SMs idle, one
 * for 128-column tiles); GDN2_STATE_LOOKAHEAD=0 selects the plain state
 * kernel for both, =64 for the 128-column tiles only (diagnostics; same
 * results up to rounding).
 *
 * Every launch after the first is a programmatic dependent launch on
 * `stream`: it may be scheduled while the kernel before it drains and waits
 * in-kernel for that kernel's results, so the call has no launch gaps.  The
 * first launch follows the stream's earlier work in the usual order.
 * GDN2_PDL=0 makes every launch a plain one (diagnostics; same results).
 */
GDN2_API gdn2_status gdn2_chunk_fwd(const void *q, const void *k, const void *v, const void *g,
                           const void *beta, const void *w, float scale,
                           const void *initial_state, const void *cu_seqlens, void *out,
                           void *final_state, const gdn2_dims *dims, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Same as gdn2_chunk_fwd, and additionally records caller-created CUDA events
 * (cudaEvent_t passed as void*) on `stream` at the boundaries of the launch
 * sequence: events[i] just before stage i and events[n_stages] after the
 * last, where n_stages = gdn2_num_stages(dims) and n_events must be at least
 * n_stages + 1 (else GDN2_ERR_NULL).  Used to time each kernel on the stream
 * it runs on.  Stage names: gdn2_stage_name.
 */
GDN2_API gdn2_status gdn2_chunk_fwd_staged(const void *q, const void *k, const void *v, const void *g,
                                           const void *beta, const void *w, float scale,
                                           const void *initial_state, const void *cu_seqlens,
                                           void *out, void *final_state, const gdn2_dims *dims,
                                           void *workspace, size_t workspace_bytes, void *stream,
                                           void *const *events, int32_t n_events);

/* Number of timed stages of the launch sequence for `dims` (0 if invalid).
 * Host-only. */
GDN2_API int32_t gdn2_num_stages(const gdn2_dims *dims);

/* Static name of stage i ("prep", "intra", ...), NULL if out of range.
 * Host-only. */
GDN2_API const char *gdn2_stage_name(const gdn2_dims *dims, int32_t i);

/* Number of kernel launches one gdn2_chunk_fwd call makes for `dims` when g
 * is given (0 if invalid); without g the tensor-core path makes one fewer
 * (no exact pass of the intra kernel).  Host-only. */
GDN2_API int32_t gdn2_launch_count(const gdn2_dims *dims);

/*
 * The launch sequence gdn2_chunk_fwd runs for `dims` on a GPU with
 * `sm_count` SMs (<= 0: 152, a GB300), as one line of text: each launch,
 * its grid, the state-pass tile width and segments, the workspace size.
 * Writes at most `len` bytes including the terminating NUL into `buf` (buf
 * may be NULL with len 0) and returns the full length, as snprintf does; 0
 * if dims is NULL or invalid.  Host-only.  With the environment variable
 * GDN2_LOG=1, gdn2_chunk_fwd prints the same line to stderr at each call.
 */
GDN2_API int32_t gdn2_launch_plan(const gdn2_dims *dims, int32_t sm_count, char *buf, size_t len);

/*
 * Workspace bytes of gdn2_recurrent_fwd for `dims` (a 64-byte status area; 0
 * if the shape is unsupported).  Host-only.
 */
GDN2_API size_t gdn2_recurrent_workspace_bytes(const gdn2_dims *dims);

/*
 * Token-by-token GDN-2 recurrence from a carried state: decode steps and short
 * continuations of a prefill (FlashGDN-2 README quick start: prefill, then
 * decode from the returned state).  Per token, the FlashInfer docs'
 * recurrence (chunk_gated_delta_rule2, op description): decay by e^{g},
 * erase read with beta, write with w, output after the write.
 *
 * Arguments, layouts, defaults and errors are those of gdn2_chunk_fwd, with
 * two differences: `workspace` needs only gdn2_recurrent_workspace_bytes
 * (the status words read by gdn2_device_status), and `final_state` may be the
 * same pointer as `initial_state` (the state is updated in place; any other
 * overlap is GDN2_ERR_ALIAS).  dims->impl is ignored.  Each token costs a
 * pass over the state held on chip; the state is read and written once per
 * call, so the call suits few tokens per sequence (gdn2_chunk_fwd is the
 * prefill path; measured on a GB300 with 128 sequences and 32 heads of 128
 * channels, the chunked call is the faster one from about 20 tokens per
 * sequence on).  Two launches: a cu_seqlens check, then one CTA per
 * (sequence, value head, 32 value columns).
 */
GDN2_API gdn2_status gdn2_recurrent_fwd(const void *q, const void *k, const void *v, const void *g,
                                        const void *beta, const void *w, float scale,
                                        const void *initial_state, const void *cu_seqlens, void *out,
                                        void *final_state, const gdn2_dims *dims, void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * Read the device-side status that the last gdn2_chunk_fwd or
 * gdn2_recurrent_fwd on this workspace wrote into *status: GDN2_OK,
 * GDN2_ERR_CU_SEQLENS, GDN2_ERR_TIMEOUT (a tensor-core kernel waited more
 * than 2 s on one of its own barriers and unwound), GDN2_ERR_RANGE (an fp16
 * intermediate was clipped) or, in a checked build only, GDN2_ERR_BOUNDS (an
 * index check failed); with any of the last three the outputs are invalid.
 * If several apply, the first in that order is reported.  This call
 * SYNCHRONISES `stream`.  Returns GDN2_ERR_CUDA if the copy fails.
 */
GDN2_API gdn2_status gdn2_device_status(const void *workspace, void *stream, int32_t *status);

/*
 * Size of the device scratch array behind gdn2_chunk_fwd_noalloc: 64 MiB,
 * enough for any problem with gdn2_workspace_bytes(dims) <= this value (for
 * example T_tot = 2048 tokens on 16 value heads of size 128, or the 256-token,
 * 2-head, size-64 case with room to spare).
 */
#define GDN2_NOALLOC_SCRATCH_BYTES 67108864u

/*
 * gdn2_chunk_fwd without a workspace argument, for callers that cannot
 * allocate device memory: code that runs where allocation is not allowed or
 * not available (a framework hook or plugin with no access to an allocator,
 * a runtime that forbids cudaMalloc after start-up) but still passes its own
 * inputs and outputs.  The paper has no counterpart; this is a packaging of
 * the same computation.
 *
 * The workspace is a fixed array of GDN2_NOALLOC_SCRATCH_BYTES inside this
 * library (a __device__ variable, so every GPU that loads the library holds
 * it until the process exits).  This call allocates nothing and calls no
 * allocating routine.  Its first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  Later calls reuse the address.
 *
 * All calls share the one array and it keeps the last call's contents; every
 * call rewrites what it reads (the status words, chunk map and chunk records
 * are written before use), so nothing needs clearing between calls.  Calls
 * that overlap on the GPU (different streams, or different host threads
 * without ordering) race on the array and must not be issued.
 *
 * Arguments and results are those of gdn2_chunk_fwd.  Returns
 * GDN2_ERR_NOALLOC_LIMIT, before touching the device, when
 * gdn2_workspace_bytes(dims) exceeds GDN2_NOALLOC_SCRATCH_BYTES;
 * GDN2_ERR_ARCH, before the address lookup, on a device that is not compute
 * capability 10.3; GDN2_ERR_CUDA if the device address cannot be looked up.
 * The looked-up address belongs to the CUDA context current at the first
 * call; it does not survive cudaDeviceReset of that device (a later call in
 * a new context would use a stale address), so do not reset a device between
 * calls.  The device-side status of the last call (cu_seqlens, timeout,
 * range) is read with gdn2_noalloc_device_status.
 */
GDN2_API gdn2_status gdn2_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *g,
                                            const void *beta, const void *w, float scale,
                                            const void *initial_state, const void *cu_seqlens, void *out,
                                            void *final_state, const gdn2_dims *dims, void *stream);

/*
 * gdn2_device_status for gdn2_chunk_fwd_noalloc: reads the status words that
 * the last gdn2_chunk_fwd_noalloc call on the current device left in the
 * library's scratch array (that call's caller has no workspace pointer to
 * pass).  Same results and the same stream SYNCHRONISATION as
 * gdn2_device_status; GDN2_ERR_ARCH or GDN2_ERR_CUDA as
 * gdn2_chunk_fwd_noalloc.  Allocates nothing.
 */
GDN2_API gdn2_status gdn2_noalloc_device_status(void *stream, int32_t *status);

/*
 * Self-test of the device-side failure detection.  Every wait in the
 * tensor-core kernels is bounded in wall time; a wait that runs out records
 * GDN2_ERR_TIMEOUT in the workspace status word and the kernel returns, so
 * the CUDA context stays usable.  This call launches one small kernel that
 * waits, through the same bounded wait, on a barrier that nothing completes,
 * for limit_ns nanoseconds (1 000 .. 100 000 000), then records the timeout.
 * Afterwards gdn2_device_status(workspace) reports GDN2_ERR_TIMEOUT.
 *   workspace        device buffer of at least 64 bytes (its status words are
 *                    overwritten); workspace_bytes its size
 * Returns GDN2_ERR_NULL / GDN2_ERR_WORKSPACE / GDN2_ERR_SHAPE (limit out of
 * range) / GDN2_ERR_ARCH before any launch, else GDN2_OK once enqueued.
 */
GDN2_API gdn2_status gdn2_selftest_wait_timeout(void *workspace, size_t workspace_bytes, uint64_t limit_ns,
                                                void *stream);

/* Static, human-readable text for a status code.  Host-only. */
GDN2_API const char *gdn2_status_string(int status);

/* Library ABI version: (major << 16) | minor.  Host-only. */
GDN2_API int32_t gdn2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN2_H */
