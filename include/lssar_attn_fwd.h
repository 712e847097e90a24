/*
 * lssar_attn_fwd.h -- C ABI of the GB300 (sm_103a) causal LSSAR attention forward.
 *
 * The operation is the attention forward defined in the papernotes.org notes on
 * "Softplus Attention with Re-weighting Boosts Length Extrapolation in Large
 * Language Models" (arXiv 2501.13428):
 *
 *   Key design 1 (LSSA): q_i <- q_i/||q_i||_2, k_j <- k_j/||k_j||_2,
 *       A_ij = Softplus(ln d * ln i * q_i.k_j) for j <= i (0 above the diagonal,
 *       a multiplicative mask applied after the Softplus), then each row of A is
 *       divided by its sum.  i is the 1-based row index (tokens attended).
 *   Key design 2 (re-weighting): A_ij <- max(i*A_ij - O_i, 0)^p with O_i = 0 for
 *       rows 1..3 and 1 otherwise, then each row is divided by its sum again.
 *   The output row i is sum_j A_ij v_j.
 *   Background (softmax mode): A = Softmax(q.k^T / sqrt(d) + causal -inf mask).
 *   Ablation table (modes 3, 4): re-weighting applied to the softmax attention
 *       above, and to LSSA with Sigmoid(x) = 1/(1+e^-x) in place of Softplus.
 *
 * A re-weighted row whose entries are all zero (possible only when the LSSA
 * row is exactly uniform) is 0/0 in the notes; this library returns the
 * uniform prefix mean for it.  Norms are clamped at 1e-12.
 *
 * Conventions shared by every entry point:
 *   - q, k, v, out are DEVICE pointers to bfloat16 tensors of shape
 *     [B, H, L, d], contiguous (d fastest), each 16-byte aligned.  The caller
 *     owns them; out must not overlap q, k or v.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and return
 *     once the work is enqueued.  Errors in the arguments are reported before
 *     anything is launched; nothing is written to `out` in that case.
 *   - Temporary device memory is taken stream-ordered from a memory pool owned
 *     by the library and released stream-ordered on the same stream.
 *   - Thread-safe: no mutable global state besides the lazily created pool
 *     (guarded) and the device error word (see lssar_device_error_word).
 *   - The device addresses of the library's own device variables (the error
 *     word, the fixed scratch of lssar_attn_fwd_noalloc) and its memory pool
 *     are looked up once per device and kept: after cudaDeviceReset (or any
 *     other teardown of a device's primary context) the library must not be
 *     used on that device again in the same process.
 */
#ifndef LSSAR_ATTN_FWD_H
#define LSSAR_ATTN_FWD_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same types as the CUDA runtime's cudaStream_t and cudaEvent_t. */
typedef struct CUstream_st *cudaStream_t;
typedef struct CUevent_st *cudaEvent_t;

typedef enum {
    LSSAR_MODE_SOFTMAX = 0,    /* Softmax(q.k^T/sqrt(d)) on raw q, k (Background)    */
    LSSAR_MODE_LSSA = 1,       /* Key design 1 only                                   */
    LSSAR_MODE_LSSAR = 2,      /* Key design 1 followed by Key design 2               */
    LSSAR_MODE_SOFTMAX_RW = 3, /* ablation: Softmax(q.k^T/sqrt(d)), then Key design 2 */
    LSSAR_MODE_SIGMOID_RW = 4  /* ablation: Key design 1 with Sigmoid in place of
                                  Softplus, then Key design 2                         */
} lssar_mode_t;

typedef enum {
    LSSAR_OK = 0,
    LSSAR_ERR_NULL = -1,    /* a tensor pointer is NULL                               */
    LSSAR_ERR_SHAPE = -2,   /* B, H or L < 1, L > 2^24, or B*H*L*d beyond 2^40         */
    LSSAR_ERR_HEADDIM = -3, /* d is not 64 or 128                                     */
    LSSAR_ERR_P = -4,       /* re-weighting mode (2, 3, 4) with p < 1 or p > 1024     */
    LSSAR_ERR_MODE = -5,    /* unknown mode                                           */
    LSSAR_ERR_ALIGN = -6,   /* a pointer is not 16-byte aligned                       */
    LSSAR_ERR_CUDA = -7,    /* a CUDA call failed (launch, pool allocation, ...)      */
    LSSAR_ERR_ALIAS = -8,   /* an output overlaps an input (or another output)         */
    LSSAR_ERR_SCRATCH = -9  /* lssar_attn_fwd_noalloc: problem needs more scratch than
                               LSSAR_NOALLOC_SCRATCH_BYTES                            */
} lssar_status_t;

/*
 * Causal attention forward, computed by the tensor-core (tcgen05/TMEM/TMA)
 * kernel for sm_103a.
 *   q, k, v : [B, H, L, d] bfloat16, device, read only.
 *   out     : [B, H, L, d] bfloat16, device, written (row i of head (b, h)).
 *   p       : integer exponent of the re-weighting (modes 2, 3, 4: 1..1024;
 *             ignored in modes 0, 1).
 *   mode    : lssar_mode_t.
 * Returns LSSAR_OK or a negative lssar_status_t.
 * Numerics of LSSAR mode with p >= 4: the weight pass evaluates the softplus
 * of a row as z + 2^-|z| / ln 2 (one exponential, z = log2(e) x) instead of
 * log2(1 + 2^z) when a bound computed from the row's statistics (its
 * threshold, spread, length and p) guarantees that the row's weights change
 * in sum by at most 2e-4 of their total (the output by at most 4e-4 max|v|);
 * other rows keep log2(1 + 2^z).  Setting LSSAR_EXACT_WEIGHTS=1 in the
 * environment keeps every row on log2(1 + 2^z) (read at each call).
 */
int lssar_attn_fwd(const void *q, const void *k, const void *v, void *out,
                   int B, int H, int L, int d, int p, int mode, cudaStream_t stream);

/*
 * lssar_attn_fwd with one re-weighting exponent per head: head h (of every
 * batch entry) uses p_per_head[h].  The notes leave an adaptive or learnable p
 * open (Limitations: p = 15 is empirical; Key findings: the best sparsity
 * depends on the length); a per-head p is what such a model needs at
 * inference time.
 *   p_per_head : HOST array of H ints, each in 1..1024, read before return.
 *   mode       : a re-weighting mode (2, 3 or 4); other modes return
 *                LSSAR_ERR_P.  H must be at most 256 (LSSAR_ERR_P otherwise).
 * Other arguments, results and errors as lssar_attn_fwd.
 */
int lssar_attn_fwd_heads_p(const void *q, const void *k, const void *v, void *out,
                           int B, int H, int L, int d, const int *p_per_head, int mode,
                           cudaStream_t stream);

/*
 * Training forward: lssar_attn_fwd that also saves, per query row, what the
 * backward pass needs (the notes train GPT-2 models with this attention).
 *   stats : [B, H, L, 4] float32, device, 16-byte aligned, written:
 *           {m, kappa, beta, W} per row, in the kernel's log2 units
 *           (z = log2(e) * x):  phi(z) = log2(1 + 2^z) (LSSA/LSSAR),
 *           2^(z - m) (softmax normalisers), 1/(1 + 2^-z) (sigmoid); the row's
 *           weights are w = max(phi kappa + beta, 0)^p with W = sum_j w
 *           (kappa = 1, beta = 0, p = 1 without re-weighting).  A row read as
 *           the uniform prefix mean has kappa = 0, beta = 1, W = i.
 * Must not overlap q, k, v or out.  Other arguments, results and errors as
 * lssar_attn_fwd (LSSAR_ERR_NULL for a NULL stats, LSSAR_ERR_ALIGN, ALIAS).
 */
int lssar_attn_fwd_train(const void *q, const void *k, const void *v, void *out, float *stats,
                         int B, int H, int L, int d, int p, int mode, cudaStream_t stream);

/*
 * Backward pass on the tensor cores: gradients of sum(dout * out) with
 * respect to q, k and v, from the row statistics of lssar_attn_fwd_train.
 * Same operation, arguments, results and errors as lssar_attn_bwd_simt below.
 * Two persistent tcgen05 kernels: a pass over each 128-query tile (dq, and the
 * per-query terms D_i = dout_i . out_i and the re-weighting threshold's
 * gradient) and a pass over each 128-key tile (dk, dv), each applying the
 * gradient of the L2 row normalisation to its own tile before it writes;
 * scores use fp16 normalised rows as in the forward, the gradient products
 * fp16 (normalised modes) or bf16 (softmax modes) with fp32 accumulation.
 * Scratch: 256 + round_up(4*B*H, 256) + 2*round_up(2*B*H*L*d, 256)
 * (normalised modes only) + round_up(32*B*H*ceil(L/128)*128, 256) bytes from
 * the library's stream-ordered pool.
 */
int lssar_attn_bwd(const void *q, const void *k, const void *v, const void *dout,
                   const float *stats, void *dq, void *dk, void *dv,
                   int B, int H, int L, int d, int p, int mode, cudaStream_t stream);

/*
 * Training with one re-weighting exponent per head (the notes leave an
 * adaptive or learnable p open: Limitations; training is where such a p would
 * be chosen).  lssar_attn_fwd_train_heads_p is lssar_attn_fwd_train, and
 * lssar_attn_bwd_heads_p is lssar_attn_bwd, with head h (of every batch entry)
 * using p_per_head[h]; pass the same array to both.
 *   p_per_head : HOST array of H ints, each in 1..1024, read before return.
 *   mode       : a re-weighting mode (2, 3 or 4); other modes return
 *                LSSAR_ERR_P.  H must be at most 256 (LSSAR_ERR_P otherwise).
 * Other arguments, results and errors as lssar_attn_fwd_train / lssar_attn_bwd.
 */
int lssar_attn_fwd_train_heads_p(const void *q, const void *k, const void *v, void *out, float *stats,
                                 int B, int H, int L, int d, const int *p_per_head, int mode,
                                 cudaStream_t stream);
int lssar_attn_bwd_heads_p(const void *q, const void *k, const void *v, const void *dout,
                           const float *stats, void *dq, void *dk, void *dv,
                           int B, int H, int L, int d, const int *p_per_head, int mode,
                           cudaStream_t stream);

/*
 * Backward pass: gradients of sum(dout * out) with respect to q, k and v,
 * given the row statistics of the forward (lssar_attn_fwd_train with the same
 * q, k, v, B, H, L, d, p, mode).  Chain rule through the steps of Key designs
 * 1-2: the derivative of the L1 normalisations, of the re-weighting threshold
 * (its row sum S1), of softplus / sigmoid / exp and of the L2 row
 * normalisation; a uniform row passes no gradient to its scores.  The
 * forward's output is not needed: dout_i . out_i is formed from the
 * recomputed weights, free of the output's bf16 rounding.
 *   q, k, v, dout : [B, H, L, d] bfloat16, device, read only.
 *   stats         : [B, H, L, 4] float32 from lssar_attn_fwd_train.
 *   dq, dk, dv    : [B, H, L, d] bfloat16, device, written; they must not
 *                   overlap each other or any input (LSSAR_ERR_ALIAS).
 * Scratch (8*B*H*L bytes) comes from the library's stream-ordered pool.  Other
 * arguments and errors as lssar_attn_fwd.
 *
 * This entry point runs a plain CUDA-core implementation (one warp per query
 * row for dq, one warp per key row for dk and dv, fp32, libm
 * transcendentals); it is the cross-check for the tensor-core backward.
 */
int lssar_attn_bwd_simt(const void *q, const void *k, const void *v, const void *dout,
                        const float *stats, void *dq, void *dk, void *dv,
                        int B, int H, int L, int d, int p, int mode, cudaStream_t stream);

/*
 * Decode step: the forward for ONE new query row per head, at position L
 * (1-based, i.e. it attends to all L cached tokens, itself included), for
 * every mode above.  Equal to row L of lssar_attn_fwd on the full sequence
 * (the notes evaluate a model trained at 1K tokens at 2K-8K: this is that
 * inference step).
 *   q       : [B, H, d] bfloat16, device (the new token's query).
 *   k_cache : [B, H, L, d] bfloat16, device (keys 1..L, the new one last).
 *   v_cache : [B, H, L, d] bfloat16, device.
 *   out     : [B, H, d] bfloat16, device, written.
 * Bound by HBM: K and V are read once.  Each head's cache is cut into up to
 * 16 chunks of at most 4096 keys that form one thread-block cluster: the
 * chunks' statistics and partial outputs meet in distributed shared memory
 * and the scores stay in shared memory, so a step is one launch that touches
 * no other global memory.  Longer caches (over 65536 keys per head) take a
 * cooperative launch with a grid barrier, or three launches when that grid
 * cannot be resident at once; those paths keep scores and partials in a
 * float scratch of about 4*B*H*L bytes from the library's pool.  The
 * environment variable LSSAR_DECODE_PATH=grid (or split) makes a call skip
 * the cluster path (or use the three launches), to test those paths at small
 * sizes.  Same errors as lssar_attn_fwd.
 */
int lssar_attn_decode(const void *q, const void *k_cache, const void *v_cache, void *out,
                      int B, int H, int L, int d, int p, int mode, cudaStream_t stream);

/*
 * Same operation and contract as lssar_attn_fwd, computed by a plain CUDA-core
 * kernel (one warp per query row, fp32 throughout, accurate libm softplus).
 * It is a second, independent GPU implementation kept for cross-checking the
 * tensor-core kernel; it is not tuned for speed.
 */
int lssar_attn_fwd_simt(const void *q, const void *k, const void *v, void *out,
                        int B, int H, int L, int d, int p, int mode, cudaStream_t stream);

/*
 * lssar_attn_fwd with timing hooks: records `ev_start` on `stream` before the
 * first kernel of the call (the normalisation prologue, LSSA/LSSAR modes),
 * `ev_main` just before the attention kernel and `ev_end` after it.  Any event
 * may be NULL (not recorded).  Events are created and owned by the caller.
 * Used by the benchmark to time the attention kernel alone; the computation
 * is identical to lssar_attn_fwd.  A non-NULL ev_main costs time: the
 * attention kernel is launched as a programmatic dependent of the prologue
 * (its launch and setup overlap the prologue's tail), and an event recorded
 * between the two makes it wait for the prologue to finish first (about 5 us
 * per call on GB300).
 */
int lssar_attn_fwd_profiled(const void *q, const void *k, const void *v, void *out,
                            int B, int H, int L, int d, int p, int mode, cudaStream_t stream,
                            cudaEvent_t ev_start, cudaEvent_t ev_main, cudaEvent_t ev_end);

/*
 * Size of the fixed device scratch array used by lssar_attn_fwd_noalloc
 * (32 MiB).  Every GPU on which the library is loaded holds it until the
 * process exits.
 */
#define LSSAR_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * lssar_attn_fwd without any device memory allocation.
 *
 * The notes on the method have no counterpart of this: it exists for callers
 * that cannot let a library allocate device memory while it runs -- for
 * example inference-runtime plugins whose execute/enqueue step is not allowed
 * to allocate, hosts that reserve their whole memory budget up front, and
 * latency-critical loops where an allocation could block on the driver.
 *
 * Same operation, arguments and results as lssar_attn_fwd.  The caller still
 * provides q, k, v and out; the temporary data (a work counter and the
 * normalised q and k in fp16: 256 + 2*round_up(2*B*H*L*d, 256) bytes in
 * LSSA/LSSAR mode, 256 bytes in softmax mode) lives in one fixed device array of
 * LSSAR_NOALLOC_SCRATCH_BYTES compiled into the library.  Problems that need
 * more return LSSAR_ERR_SCRATCH before anything is launched (for example
 * B*H*L*d must stay below about 8.4 million elements in LSSA/LSSAR mode).
 * No cudaMalloc, cudaFree or pool allocation is made.
 *
 * The first call on a device looks up that device's copy of the array (and
 * may make the CUDA driver load the library's device code); make that first
 * call before any stream capture.  All calls share the one array per device
 * and it keeps the previous call's contents; the parts that must start at zero
 * are cleared by each call on its stream.  Calls whose execution overlaps on
 * the GPU (different streams, or different host threads, without ordering
 * between them) race on the array: order them.  The device address of the
 * array is looked up once per device and kept: do not use the library on a
 * device after cudaDeviceReset (or any other teardown of its primary context)
 * in the same process.
 */
int lssar_attn_fwd_noalloc(const void *q, const void *k, const void *v, void *out,
                           int B, int H, int L, int d, int p, int mode, cudaStream_t stream);

/*
 * Introspection of the attention kernel's work schedule (host only, no CUDA
 * call).  Work items are pairs of 128-row Q tiles of one head, numbered
 * longest first (item i: head i % BH, pair n_pairs - 1 - i / BH).  CTA c of a
 * grid of `grid` CTAs first processes first[2c] and then first[2c+1] (-1:
 * none), then the items from *tail_base on, as a global counter hands them
 * out.  first must hold 2*grid ints; 1 <= grid <= 256.  Returns LSSAR_OK,
 * LSSAR_ERR_NULL or LSSAR_ERR_SHAPE.
 */
int lssar_schedule_plan(int BH, int n_qtiles, int grid, int *first, int *tail_base);

/*
 * The launch plan of lssar_attn_decode for these sizes on the current device
 * (host only: queries the device's SM count and occupancy, launches nothing).
 * Outputs, each may be NULL: *path = 0 (one launch, a thread-block cluster per
 * head), 1 (one cooperative launch) or 2 (three launches); *launches = the
 * kernel launches one decode call makes (1, 1 or 3); *chunks = pieces of
 * each head's cache; *chunk_rows = keys per piece (the last one shorter).
 * The environment variable LSSAR_DECODE_PATH is honoured as by the call.
 * Returns LSSAR_OK, LSSAR_ERR_SHAPE / LSSAR_ERR_HEADDIM on sizes the call
 * rejects, or LSSAR_ERR_CUDA (no device).
 */
int lssar_decode_plan(int B, int H, int L, int d, int *path, int *launches, int *chunks, int *chunk_rows);

/*
 * TEST ONLY: the failure path of the bounded waits.  Runs one decode step
 * (B=1 H=4 L=512 d=64, zero inputs, internal scratch) whose producer warps
 * withhold every copy, so that each wait of that launch gives up after its
 * 2 s bound: the kernel records decode code 41 in the device error word,
 * leaves its loops and ends without a fault (no copy is in flight).  Takes
 * about 2 s on the GPU; returns LSSAR_OK once launched, LSSAR_ERR_CUDA
 * otherwise.  Read the code with lssar_device_error_word afterwards.
 */
int lssar_selftest_stall(cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *lssar_status_string(int status);

/*
 * Reads and clears the device error word of the current device: 0 when no
 * kernel of this library has hit a bounded wait since the last call, else a
 * code (1-based pipeline stage) of the first wait that gave up.  Synchronises
 * the current device.  Returns LSSAR_OK or LSSAR_ERR_CUDA.
 */
int lssar_device_error_word(unsigned int *word);

/* Version of this ABI: major * 10000 + minor * 100 + patch. */
int lssar_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LSSAR_ATTN_FWD_H */
