/*
 * ttt.h -- C ABI of the TTT inner-loop library (libttt.so).
 *
 * The method (TTT layer, mini-batch form: forward, decode step, and the TTT-Linear
 * backward pass).  Per (batch, head) a
 * fast-weight state is trained while the sequence is read:
 *   - update/apply recurrence: W_t = W_{t-1} - eta_t grad_W l(W_{t-1}; x_t),
 *     o_t = f(q_t; W_t)  -- damodev.csdn.net TTT article, section 3.1, equation;
 *     the output uses the weights after the token's own update;
 *   - mini-batch TTT: inside each mini-batch of b tokens every gradient is taken
 *     at the mini-batch's starting weights, and the state reached at the end of
 *     the mini-batch is carried to the next one -- same article, sections 4.1-4.2;
 *   - loss l = 1/2 || f(k_t) - v_t ||^2 (summed over features, no 1/d);
 *   - TTT-Linear f(k) = k W + c with W [d, d] row-major and c [d] -- same article,
 *     sections 4.2 (XK @ W1 + b1) and 4.3 (W1 [heads, d, d], b1 [heads, 1, d]);
 *   - TTT-MLP f(k) = GELU_tanh(k W1 + b1) W2 + b2, W1 [d, dh], W2 [dh, d] --
 *     lryc.cn TTT article, section 2.1 (d -> 4d GELU -> d);
 *   - optional residual LayerNorm f(k) = k + LN(f_res(k)) with per-head gamma,
 *     beta [H, d], biased variance and eps = ln_eps -- lryc.cn article, section 2.1;
 *     the loss target of f_res is then v - k (damodev article, section 4.2).
 * The per-token learning rate eta, the gate eta_base * sigmoid(theta_lr . x) of
 * the lryc.cn article, section 2.2, is an input of the scan entry points;
 * ttt_eta_gate computes it on the GPU from the layer's input tokens.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers (cudaMalloc or equivalent) owned
 *     by the caller.  The library allocates no memory and keeps no per-call
 *     state; it only launches kernels on `stream` and returns.  Results are
 *     valid once the stream has been synchronised (ttt_sync_status does that
 *     and also reports device-side failures).
 *   - Layouts are dense row-major, no padding, 16-byte aligned base pointers
 *     (shapes below for a call on all B*H rows; see bh_offset/bh_count):
 *       Q, K, V, Z   [B, H, L, d]   element type desc->io_dtype
 *       eta          [B, H, L]      float
 *       gamma, beta  [H, d]         float  (may be NULL iff residual_ln == 0)
 *       initial state: leading [H] (init_per_batch == 0) or [B, H]
 *       final state:   always leading [B, H]; always float.
 *   - Z must not alias any input.  A final-state buffer may alias the matching
 *     initial-state buffer only when init_per_batch == 1 (same shape).
 *   - Errors: TTT_ERR_INVALID_ARG for NULL pointers, non-positive sizes,
 *     L % mini_batch != 0, misaligned pointers or forbidden aliasing;
 *     TTT_ERR_UNSUPPORTED for shapes no kernel handles; TTT_ERR_CUDA when a
 *     CUDA call or launch fails.  Nothing is launched when an error is
 *     returned.  No C++ exception crosses this interface.  ttt_last_error()
 *     gives a one-line description of the calling thread's last failure.
 */
#ifndef TTT_H
#define TTT_H

#if defined(__GNUC__)
#define TTT_API __attribute__((visibility("default")))
#else
#define TTT_API
#endif

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *ttt_stream_t;

typedef enum {
    TTT_OK = 0,
    TTT_ERR_INVALID_ARG = 1,
    TTT_ERR_UNSUPPORTED = 2,
    TTT_ERR_CUDA = 3,
    TTT_ERR_TIMEOUT = 4 /* a device-side bounded wait gave up (see ttt_sync_status) */
} ttt_status;

typedef enum { TTT_F32 = 0, TTT_BF16 = 1 } ttt_dtype;

typedef struct {
    int B;              /* batch                                               */
    int H;              /* heads                                               */
    int L;              /* sequence length, a multiple of mini_batch           */
    int d;              /* head dimension (features of q, k, v, z)             */
    int d_hidden;       /* TTT-MLP hidden width dh; 0 means 4 d (linear: unused) */
    int mini_batch;     /* b, tokens per mini-batch                            */
    ttt_dtype io_dtype; /* element type of Q, K, V and Z; state is always float */
    int residual_ln;    /* 0: f = f_res;  1: f(k) = k + LN(f_res(k))           */
    float ln_eps;       /* LayerNorm eps, finite and > 0 when residual_ln      */
    int init_per_batch; /* 0: initial state [H, ...];  1: [B, H, ...]          */
    /* (batch, head) partition: the call covers rows bh_offset .. bh_offset + rows - 1 of
     * the flattened B*H grid (row = b*H + h), rows = bh_count (0: all B*H rows, with
     * bh_offset 0).  Every row-indexed buffer (Q, K, V, Z, eta, the final state, and
     * the initial state when init_per_batch) starts at the call's first row and holds
     * `rows` rows; head-indexed parameters (a head-shared initial state, gamma, beta)
     * are passed whole, and row i of the call uses head (bh_offset + i) mod H.  Rows
     * are independent, so calls on disjoint ranges (e.g. one per GPU) together give
     * the result of one call on all rows. */
    int bh_offset;
    int bh_count;
    /* inner learner (the design dimensions of the ai-feeds "Modular TTT" page):
     * loss TTT_LOSS_MSE (1/2 ||f(k) - v||^2, the default) or TTT_LOSS_INNER_PRODUCT
     * (-<f(k), v>); weight_decay lambda >= 0 adds 1/2 lambda ||W||^2 over the weight
     * matrices (W; W1, W2 -- not the biases) to every token's loss, taken at the
     * mini-batch's starting weights like the gradient: inside a mini-batch
     * W_t = (1 - lambda sum_{s<=t} eta_s) W_start - sum_{s<=t} eta_s grad l_s. */
    int loss;
    float weight_decay;
    /* Optional per-call failure word: a device pointer to a caller-owned, 4-byte aligned
     * unsigned int.  When it is non-NULL, the call's kernels report a bounded wait that ran
     * out by setting bit 0 of this word (atomic OR) instead of the device-wide flag that
     * ttt_sync_status reads, so callers on different streams see only their own calls'
     * failures; the caller clears it and reads it after synchronising its stream.  NULL:
     * the device-wide flag.  (Kernels without bounded waits never write it.) */
    unsigned int *status;
} ttt_desc;

enum { TTT_LOSS_MSE = 0, TTT_LOSS_INNER_PRODUCT = 1 };

/*
 * TTT-Linear forward.
 *   in : Q, K, V [B,H,L,d] (io_dtype); eta [B,H,L]; W0 [H or B,H, d, d];
 *        b0 [H or B,H, d]; gamma, beta [H, d] (NULL allowed without LN).
 *   out: Z [B,H,L,d] (io_dtype): z_t = f(q_t; W_t, c_t) with the weights after
 *        token t's update; W_final [B,H,d,d], b_final [B,H,d]: state after
 *        the last mini-batch.
 * Supported: d <= 128 with d a multiple of 4, and b <= 64 (generic kernels, fp32
 * arithmetic: without the residual LayerNorm and with at most 2 x 148 CTAs' worth of
 * (batch, head) rows, each row split over CTAs by output column, since the columns of the
 * state evolve independently there; otherwise one CTA per row); bf16 I/O with d = 64,
 * b = 16 runs a tensor-core kernel: without the residual LayerNorm the chunked kernel (the
 * state carried across 64-token chunks; every loss and decay), with it the fused kernel
 * (every loss and decay).
 */
TTT_API ttt_status ttt_linear_fwd(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                          const float *eta, const float *W0, const float *b0,
                          const float *gamma, const float *beta, void *Z, float *W_final,
                          float *b_final, ttt_stream_t stream);

/*
 * TTT-MLP forward (two-layer fast weights, GELU tanh).
 *   in : Q, K, V, eta as above; W1_0 [H or B,H, d, dh]; b1_0 [H or B,H, dh];
 *        W2_0 [H or B,H, dh, d]; b2_0 [H or B,H, d]; gamma, beta [H, d].
 *   out: Z [B,H,L,d]; W1_f [B,H,d,dh]; b1_f [B,H,dh]; W2_f [B,H,dh,d]; b2_f [B,H,d].
 * Supported: d <= 128, dh <= 512, b <= 64 while the state fits on chip; the
 * tensor-core kernel (bf16, d = 64, dh = 256, b = 16) and the generic kernel run every
 * loss and decay.  With TTT_MLP_KERNEL=tmem in the environment (read at each call), bf16
 * calls with d = 64, dh = 256, b = 16 and no weight decay run the tcgen05 kernel instead:
 * W1^T and W2 resident in tensor memory as fp32, the hidden-width products on tcgen05 (same
 * results within bf16 rounding; slower at b = 16, hence not the default).
 */
TTT_API ttt_status ttt_mlp_fwd(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                       const float *eta, const float *W1_0, const float *b1_0,
                       const float *W2_0, const float *b2_0, const float *gamma,
                       const float *beta, void *Z, float *W1_f, float *b1_f, float *W2_f,
                       float *b2_f, ttt_stream_t stream);

/*
 * TTT-Linear decode step (the state carried between calls, like a cache).
 * The desc->L tokens of every (batch, head) are processed one at a time: the
 * mini-batch form with desc->mini_batch == 1 (required), which is the per-token
 * recurrence itself.  The state is per (batch, head) and updated in place:
 *   in : Q, K, V [B,H,L,d] (io_dtype); eta [B,H,L]; gamma, beta [H, d] (NULL
 *        allowed without LN);
 *   in/out: W [B,H,d,d], b [B,H,d] (float): read as the state before the first
 *        token, overwritten with the state after the last one;
 *   out: Z [B,H,L,d] (io_dtype), z_t = f(q_t; W_t, c_t) after token t's update.
 * Calling it T times with one token each gives the same result as one call
 * with the T tokens.  desc->init_per_batch is ignored (the state is always
 * [B, H, ...]).  Supported: d <= 128 with d a multiple of 4; d = 64 runs the decode
 * kernel (FP32: one warp per (batch, head) with the residual LayerNorm, four warps of 16
 * output columns each without it, since the columns of the state then evolve
 * independently), other d the generic kernel.  Z must not alias an input, and W, b must
 * not alias any other buffer.
 */
TTT_API ttt_status ttt_linear_step(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                                   const float *eta, float *W, float *b, const float *gamma,
                                   const float *beta, void *Z, ttt_stream_t stream);

/*
 * TTT-Linear backward: the vector-Jacobian product of ttt_linear_fwd, the gradient that
 * training through the inner loop needs (the meta-learning gradient of the damodev.csdn.net
 * TTT article, section 6.1, taken through the mini-batch scan of sections 4.1-4.2, with the
 * residual LayerNorm of the lryc.cn TTT article, section 2.1).  For the outer loss
 * F = <Z, dZ> + <W_final, dW_final> + <b_final, db_final> it writes
 *   dQ, dK, dV [B,H,L,d] (io_dtype), deta [B,H,L] float,
 *   dW0 [H or B,H, d, d], db0 [H or B,H, d] float (shaped like W0, b0: with a head-shared
 *        initial state, the sum over the call's rows of each head; a head with no row in
 *        the call gets 0),
 *   dgamma, dbeta [H, d] float with the residual LayerNorm (the same per-head sums; NULL
 *        allowed without it).
 *   in : Q, K, V, dZ [B,H,L,d] (io_dtype); eta [B,H,L]; W0, b0, gamma, beta as the forward
 *        (gamma, beta NULL allowed without LN); dW_final [B,H,d,d], db_final [B,H,d]
 *        float, or NULL for zero.
 *   workspace: device memory of at least ttt_linear_bwd_workspace_size(desc) bytes,
 *        256-byte aligned, owned by the caller; the call overwrites it (state checkpoints
 *        of a forward re-run and per-row partial gradients).  Calls that share a workspace
 *        must not overlap in time.
 * Supported: with or without the residual LayerNorm, either loss, with or without weight
 * decay, d <= 128 with d a multiple of 4, b <= 64 (as far as the state checkpoints fit in
 * shared memory); fp32 arithmetic.  Otherwise TTT_ERR_UNSUPPORTED.  Outputs may overlap neither each other, the workspace
 * nor an input.
 */
TTT_API size_t ttt_linear_bwd_workspace_size(const ttt_desc *desc);   /* 0: invalid or unsupported */
TTT_API ttt_status ttt_linear_bwd(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                                  const float *eta, const float *W0, const float *b0, const float *gamma,
                                  const float *beta, const void *dZ, const float *dW_final,
                                  const float *db_final, void *dQ, void *dK, void *dV, float *deta,
                                  float *dW0, float *db0, float *dgamma, float *dbeta, void *workspace,
                                  size_t workspace_bytes, ttt_stream_t stream);

/*
 * ttt_linear_bwd on the library's own static device scratch (no counterpart on the pages:
 * an interface for callers that must not allocate device memory, e.g. a serving or
 * training process whose device memory is fixed at start-up, or a C caller without a
 * device allocator of its own).  Same arguments, results and errors as ttt_linear_bwd
 * without the workspace; it allocates nothing.  The scratch is a 64 MiB file-scope device
 * array per device (ttt_linear_bwd_static_scratch_bytes()); a call whose
 * ttt_linear_bwd_workspace_size exceeds it fails with TTT_ERR_INVALID_ARG.  Nothing in it
 * needs to start at zero.  The first call on a device, with that device current, resolves
 * the scratch address (cudaGetSymbolAddress, which may load the library's module); make it
 * before any stream capture.  All calls on a device share the one scratch: calls whose
 * execution overlaps in time (other streams, other host threads) race on it and give
 * undefined results, so serialise them (one stream, or synchronise between calls).
 */
TTT_API size_t ttt_linear_bwd_static_scratch_bytes(void);
TTT_API ttt_status ttt_linear_bwd_static(const ttt_desc *desc, const void *Q, const void *K,
                                         const void *V, const float *eta, const float *W0,
                                         const float *b0, const float *gamma, const float *beta,
                                         const void *dZ, const float *dW_final, const float *db_final,
                                         void *dQ, void *dK, void *dV, float *deta, float *dW0,
                                         float *db0, float *dgamma, float *dbeta, ttt_stream_t stream);

/*
 * Per-token learning rate (the learnable gate of the lryc.cn TTT article,
 * section 2.2): eta[b, h, t] = eta_base * sigmoid(theta[h] . x[b, t]).
 *   in : x [B, L, d_model] (x_dtype), the layer's input tokens; theta [H, d_model]
 *        float, one gate vector per head; eta_base, the base learning rate;
 *   out: eta [B, H, L] float -- the eta the scan entry points take.
 * The contraction is carried in fp32 (bf16 tokens meet theta split into two bf16
 * parts, so theta keeps ~16 mantissa bits).  bf16 tokens need d_model % 8 == 0.
 * eta must not overlap x or theta.  max_sms > 0 caps the grid at that many SMs' worth of
 * CTAs (0: every SM), so that the call can run beside a scan that holds the other SMs;
 * max_sms < 0 is TTT_ERR_INVALID_ARG.  Errors as for the other entry points; a bounded wait
 * that runs out is reported by ttt_sync_status.
 */
TTT_API ttt_status ttt_eta_gate(int B, int H, int L, int d_model, ttt_dtype x_dtype,
                                float eta_base, const void *x, const float *theta, float *eta,
                                int max_sms, ttt_stream_t stream);

/*
 * The TTT layer's input projections (the views theta_Q x, theta_K x, theta_V x of the
 * layer's input tokens, lryc.cn TTT article, section 2.2), written in the layout the scan
 * reads:
 *   Q[b, h, t, j] = sum_i x[b, t, i] W[h d + j, i],  K from rows H d + h d + j,
 *   V from rows 2 H d + h d + j.
 *   in : x [B, L, d_model] bf16; W [3 H d, d_model] bf16 (the three projection matrices
 *        stacked, one row per output unit, as a linear layer stores its weight);
 *   out: Q, K, V [B, H, L, d] bf16 (fp32 accumulation, rounded once).
 * Supported: d = 64, d_model a multiple of 64, 3 H d a multiple of 256 (tcgen05 kernel);
 * otherwise TTT_ERR_UNSUPPORTED.  x, W, Q, K, V 16-byte aligned; the outputs may overlap
 * neither each other nor an input.  max_sms > 0 caps the persistent grid at that many SMs
 * (0: every SM; the kernel runs in pairs of CTAs, so an odd cap is rounded down to an even
 * one, and a cap of 1 to one pair), for a call that runs beside a scan holding the other
 * SMs; max_sms < 0 is TTT_ERR_INVALID_ARG.  A bounded wait that runs out is reported by
 * ttt_sync_status.
 */
TTT_API ttt_status ttt_qkv_proj(int B, int H, int L, int d_model, int d, const void *x, const void *W,
                                void *Q, void *K, void *V, int max_sms, ttt_stream_t stream);

/*
 * Synchronises `stream`, then reports TTT_ERR_CUDA if a CUDA error is pending
 * and TTT_ERR_TIMEOUT if any kernel launched by this library on the stream's
 * device (the current device for the legacy default stream) since the previous
 * ttt_sync_status call gave up on a bounded wait (its outputs are then
 * unspecified).  Clears the device-side flag it read.  The flag is one word per
 * device, shared by every stream on it: a timeout on one stream is reported to
 * whichever caller synchronises first.
 */
TTT_API ttt_status ttt_sync_status(ttt_stream_t stream);

/*
 * Bound of every wait a kernel makes on an mbarrier (a copy landing, a buffer
 * being released), in nanoseconds of GPU wall time; <= 0 restores the default
 * of one second.  A wait that runs out makes the kernel stop waiting, finish
 * without faulting, and flag TTT_ERR_TIMEOUT for ttt_sync_status.  Process-wide
 * setting read at launch time.
 */
TTT_API void ttt_set_wait_timeout_ns(long long ns);

/*
 * Test hook for the timeout path: while `on` is non-zero, the fused kernels
 * issue no copies of the input stages, so every wait for data runs out after
 * the timeout above and the call reports TTT_ERR_TIMEOUT (outputs unspecified).
 * Nothing faults or hangs.  Process-wide; leave it off outside tests.
 */
TTT_API void ttt_debug_withhold_loads(int on);

/* Static, NUL-terminated name of a status code. */
TTT_API const char *ttt_status_string(ttt_status status);

/* One-line description of the calling thread's most recent failure ("" if none). */
TTT_API const char *ttt_last_error(void);

/* Name of the kernel ttt_linear_fwd / ttt_mlp_fwd would launch for `desc`
 * (is_mlp = 0 or 1), or NULL when the descriptor is rejected. */
TTT_API const char *ttt_kernel_name(const ttt_desc *desc, int is_mlp);

/* Library ABI version (major * 100 + minor); 101 added bh_offset/bh_count, 102 loss and
 * weight_decay, 103 ttt_linear_bwd, 104 its residual-LayerNorm form (gamma, beta, dgamma,
 * dbeta arguments), 105 the per-call status word (ttt_desc.status), 106 ttt_qkv_proj, 107 the
 * max_sms argument of ttt_eta_gate and ttt_qkv_proj. */
TTT_API int ttt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TTT_H */
