// ttt_api.cu -- host side of the C ABI declared in include/ttt.h: argument
// checks, kernel choice, launch on the caller's stream, status reporting.
// No allocation happens here; the only device memory the library owns is the
// 4-byte failure flag below, which the module loader places in the image.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "ttt_internal.h"

namespace {

// Set (atomicOr) by a kernel whose bounded wait gave up; read and cleared by
// ttt_sync_status.  One per device; shared by every call on that device.
__device__ unsigned int g_ttt_failure_flag;

thread_local char g_last_error[256];

ttt_status fail(ttt_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

ttt_status ok()
{
    g_last_error[0] = '\0';
    return TTT_OK;
}

}  // namespace

namespace ttt {
// Error reports of ttt_linear_bwd_static (its own translation unit), in this file's format.
ttt_status fail_static_scratch(size_t need, size_t have)
{
    return fail(TTT_ERR_INVALID_ARG, "the call needs %zu bytes of scratch, the static scratch holds %zu",
                need, have);
}
ttt_status fail_cuda(const char *what, cudaError_t e)
{
    return fail(TTT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}
}  // namespace ttt

namespace {

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void *p, size_t bytes)
{
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + bytes};
}

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

ttt_status check_desc(const ttt_desc *s, bool mlp)
{
    if (!s) return fail(TTT_ERR_INVALID_ARG, "desc is NULL");
    if (s->B <= 0 || s->H <= 0 || s->L <= 0 || s->d <= 0 || s->mini_batch <= 0)
        return fail(TTT_ERR_INVALID_ARG, "B, H, L, d and mini_batch must be positive");
    if (s->L % s->mini_batch != 0)
        return fail(TTT_ERR_INVALID_ARG, "L (%d) is not a multiple of mini_batch (%d)", s->L,
                    s->mini_batch);
    if (s->io_dtype != TTT_F32 && s->io_dtype != TTT_BF16)
        return fail(TTT_ERR_INVALID_ARG, "io_dtype must be TTT_F32 or TTT_BF16");
    if (s->residual_ln != 0 && s->residual_ln != 1)
        return fail(TTT_ERR_INVALID_ARG, "residual_ln must be 0 or 1");
    if (s->init_per_batch != 0 && s->init_per_batch != 1)
        return fail(TTT_ERR_INVALID_ARG, "init_per_batch must be 0 or 1");
    if (s->residual_ln && !(std::isfinite(s->ln_eps) && s->ln_eps > 0.f))
        return fail(TTT_ERR_INVALID_ARG, "ln_eps must be finite and > 0 with the residual LayerNorm");
    if (mlp && s->d_hidden < 0) return fail(TTT_ERR_INVALID_ARG, "d_hidden must be >= 0");
    if ((long long)s->B * s->H > 0x7fffffffLL)
        return fail(TTT_ERR_INVALID_ARG, "B * H exceeds the grid limit");
    if (s->loss != TTT_LOSS_MSE && s->loss != TTT_LOSS_INNER_PRODUCT)
        return fail(TTT_ERR_INVALID_ARG, "loss must be TTT_LOSS_MSE or TTT_LOSS_INNER_PRODUCT");
    if (!(std::isfinite(s->weight_decay) && s->weight_decay >= 0.f))
        return fail(TTT_ERR_INVALID_ARG, "weight_decay must be finite and >= 0");
    if (s->bh_offset < 0 || s->bh_count < 0)
        return fail(TTT_ERR_INVALID_ARG, "bh_offset and bh_count must be >= 0");
    if (s->bh_count == 0 && s->bh_offset != 0)
        return fail(TTT_ERR_INVALID_ARG, "bh_offset needs bh_count > 0");
    if ((long long)s->bh_offset + s->bh_count > (long long)s->B * s->H)
        return fail(TTT_ERR_INVALID_ARG, "rows [%d, %d) exceed B * H = %d", s->bh_offset,
                    s->bh_offset + s->bh_count, s->B * s->H);
    if (reinterpret_cast<uintptr_t>(s->status) % alignof(unsigned int) != 0)
        return fail(TTT_ERR_INVALID_ARG, "status must be 4-byte aligned");
    return TTT_OK;
}

ttt_status check_ptr(const void *p, const char *name)
{
    if (!p) return fail(TTT_ERR_INVALID_ARG, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
        return fail(TTT_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return TTT_OK;
}

constexpr int kMaxDevices = 64;

// Pointer to this device's failure flag, looked up once per device.  Host threads may race
// on the first lookup; each entry is an atomic, and every racer stores the same address.
unsigned int *failure_flag(ttt_status *st)
{
    static std::atomic<unsigned int *> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *st = fail(TTT_ERR_CUDA, "cudaGetDevice failed");
        return nullptr;
    }
    unsigned int *flag = cache[dev].load(std::memory_order_acquire);
    if (!flag) {
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_ttt_failure_flag);
        if (e != cudaSuccess) {
            *st = fail(TTT_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            return nullptr;
        }
        flag = static_cast<unsigned int *>(ptr);
        cache[dev].store(flag, std::memory_order_release);
    }
    *st = TTT_OK;
    return flag;
}

const char *linear_kernel(const ttt_desc &s)
{
    if (ttt::linear_chunk_supported(s)) return "ttt_linear_chunked";
    if (ttt::linear_tc_supported(s)) return "ttt_linear_fused";
    if (ttt::linear_cols_dc(s)) return "ttt_linear_cols";
    if (ttt::linear_generic_smem_bytes(s)) return "ttt_linear_generic";
    return nullptr;
}

constexpr const char *kMlpTmem = "ttt_mlp_tmem", *kMlpFused = "ttt_mlp_fused";

// TTT_MLP_KERNEL=tmem in the environment selects the tcgen05 kernel (fast weights in tensor
// memory) where it applies; by default the warp-MMA kernel runs, which is faster at b = 16.
bool mlp_tmem_requested()
{
    const char *v = std::getenv("TTT_MLP_KERNEL");
    return v && std::strcmp(v, "tmem") == 0;
}

const char *mlp_kernel(const ttt_desc &s)
{
    if (ttt::mlp_tmem_supported(s) && mlp_tmem_requested()) return kMlpTmem;
    if (ttt::mlp_tc_supported(s)) return kMlpFused;
    if (ttt::mlp_generic_smem_bytes(s)) return "ttt_mlp_generic";
    return nullptr;
}

}  // namespace

extern "C" {

int ttt_version(void) { return 107; }

const char *ttt_status_string(ttt_status s)
{
    switch (s) {
    case TTT_OK: return "TTT_OK";
    case TTT_ERR_INVALID_ARG: return "TTT_ERR_INVALID_ARG";
    case TTT_ERR_UNSUPPORTED: return "TTT_ERR_UNSUPPORTED";
    case TTT_ERR_CUDA: return "TTT_ERR_CUDA";
    case TTT_ERR_TIMEOUT: return "TTT_ERR_TIMEOUT";
    }
    return "TTT_ERR_UNKNOWN";
}

const char *ttt_last_error(void) { return g_last_error; }

const char *ttt_kernel_name(const ttt_desc *desc, int is_mlp)
{
    if (check_desc(desc, is_mlp != 0) != TTT_OK) return nullptr;
    if (is_mlp) {
        ttt_desc s = *desc;
        if (s.d_hidden == 0) s.d_hidden = 4 * s.d;
        return mlp_kernel(s);
    }
    return linear_kernel(*desc);
}

ttt_status ttt_linear_fwd(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                          const float *eta, const float *W0, const float *b0,
                          const float *gamma, const float *beta, void *Z, float *W_final,
                          float *b_final, ttt_stream_t stream)
{
    ttt_status st = check_desc(desc, false);
    if (st != TTT_OK) return st;
    const ttt_desc &s = *desc;
    const void *ptrs[] = {Q, K, V, eta, W0, b0, Z, W_final, b_final};
    const char *names[] = {"Q", "K", "V", "eta", "W0", "b0", "Z", "W_final", "b_final"};
    for (int i = 0; i < 9; ++i)
        if ((st = check_ptr(ptrs[i], names[i])) != TTT_OK) return st;
    if (s.residual_ln) {
        if ((st = check_ptr(gamma, "gamma")) != TTT_OK) return st;
        if ((st = check_ptr(beta, "beta")) != TTT_OK) return st;
    }
    const size_t es = s.io_dtype == TTT_BF16 ? 2 : 4;
    const size_t BH = (size_t)ttt::call_rows(s), ninit = s.init_per_batch ? BH : (size_t)s.H;
    const size_t dd = (size_t)s.d * s.d;
    const Range rq = range_of(Q, BH * s.L * s.d * es), rk = range_of(K, BH * s.L * s.d * es),
                rv = range_of(V, BH * s.L * s.d * es), re = range_of(eta, BH * s.L * 4),
                rw0 = range_of(W0, ninit * dd * 4), rb0 = range_of(b0, ninit * s.d * 4),
                rz = range_of(Z, BH * s.L * s.d * es), rwf = range_of(W_final, BH * dd * 4),
                rbf = range_of(b_final, BH * s.d * 4);
    Range ins[] = {rq, rk, rv, re, rw0, rb0, range_of(gamma, s.residual_ln ? s.H * s.d * 4 : 0),
                   range_of(beta, s.residual_ln ? s.H * s.d * 4 : 0)};
    for (const Range &r : ins)
        if (overlap(rz, r)) return fail(TTT_ERR_INVALID_ARG, "Z overlaps an input");
    if (overlap(rwf, rbf) || overlap(rz, rwf) || overlap(rz, rbf))
        return fail(TTT_ERR_INVALID_ARG, "output buffers overlap");
    for (int i = 0; i < 8; ++i) {
        const Range &r = ins[i];
        bool wf_ok = s.init_per_batch && i == 4 && r.lo == rwf.lo;  // in-place state carry
        bool bf_ok = s.init_per_batch && i == 5 && r.lo == rbf.lo;
        if (overlap(rwf, r) && !wf_ok) return fail(TTT_ERR_INVALID_ARG, "W_final overlaps an input");
        if (overlap(rbf, r) && !bf_ok) return fail(TTT_ERR_INVALID_ARG, "b_final overlaps an input");
    }
    const char *kname = linear_kernel(s);
    if (!kname)
        return fail(TTT_ERR_UNSUPPORTED, "no kernel for d=%d mini_batch=%d", s.d, s.mini_batch);

    ttt::LinearArgs a{s, Q, K, V, eta, W0, b0, gamma, beta, Z, W_final, b_final,
                      reinterpret_cast<cudaStream_t>(stream), nullptr};
    a.status = s.status ? s.status : failure_flag(&st);
    if (st != TTT_OK) return st;
    cudaError_t e = ttt::linear_chunk_supported(s) ? ttt::launch_linear_chunk(a)
                    : ttt::linear_tc_supported(s)  ? ttt::launch_linear_tc(a)
                    : ttt::linear_cols_dc(s)       ? ttt::launch_linear_cols(a)
                                                   : ttt::launch_linear_generic(a);
    if (e != cudaSuccess) return fail(TTT_ERR_CUDA, "%s launch: %s", kname, cudaGetErrorString(e));
    return ok();
}

size_t ttt_linear_bwd_workspace_size(const ttt_desc *desc)
{
    if (check_desc(desc, false) != TTT_OK) return 0;
    return ttt::linear_bwd_workspace_bytes(*desc);
}

ttt_status ttt_linear_bwd(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                          const float *eta, const float *W0, const float *b0, const float *gamma,
                          const float *beta, const void *dZ, const float *dW_final,
                          const float *db_final, void *dQ, void *dK, void *dV, float *deta,
                          float *dW0, float *db0, float *dgamma, float *dbeta, void *workspace,
                          size_t workspace_bytes, ttt_stream_t stream)
{
    ttt_status st = check_desc(desc, false);
    if (st != TTT_OK) return st;
    const ttt_desc &s = *desc;
    if (!ttt::linear_bwd_checkpoint_every(s))
        return fail(TTT_ERR_UNSUPPORTED,
                    "the backward pass takes d <= 128 (a multiple of 4) and mini_batch <= 64 "
                    "(with the state checkpoints in shared memory)");
    if (s.residual_ln) {
        const void *lp[] = {gamma, beta, dgamma, dbeta};
        const char *ln_names[] = {"gamma", "beta", "dgamma", "dbeta"};
        for (int i = 0; i < 4; ++i)
            if ((st = check_ptr(lp[i], ln_names[i])) != TTT_OK) return st;
    }
    const void *ptrs[] = {Q, K, V, eta, W0, b0, dZ, dQ, dK, dV, deta, dW0, db0, workspace};
    const char *names[] = {"Q", "K", "V", "eta", "W0", "b0", "dZ", "dQ", "dK", "dV", "deta",
                           "dW0", "db0", "workspace"};
    for (int i = 0; i < 14; ++i)
        if ((st = check_ptr(ptrs[i], names[i])) != TTT_OK) return st;
    if (dW_final && (st = check_ptr(dW_final, "dW_final")) != TTT_OK) return st;
    if (db_final && (st = check_ptr(db_final, "db_final")) != TTT_OK) return st;
    const size_t need = ttt::linear_bwd_workspace_bytes(s);
    if (workspace_bytes < need)
        return fail(TTT_ERR_INVALID_ARG, "workspace holds %zu bytes, the call needs %zu", workspace_bytes, need);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(TTT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t es = s.io_dtype == TTT_BF16 ? 2 : 4;
    const size_t BH = (size_t)ttt::call_rows(s), ninit = s.init_per_batch ? BH : (size_t)s.H;
    const size_t tok = BH * s.L * s.d, dd = (size_t)s.d * s.d;
    const size_t lnb = s.residual_ln ? (size_t)s.H * s.d * 4 : 0;
    const Range ins[] = {range_of(Q, tok * es), range_of(K, tok * es), range_of(V, tok * es),
                         range_of(eta, BH * s.L * 4), range_of(W0, ninit * dd * 4),
                         range_of(b0, ninit * s.d * 4), range_of(dZ, tok * es),
                         range_of(dW_final, dW_final ? BH * dd * 4 : 0),
                         range_of(db_final, db_final ? BH * s.d * 4 : 0),
                         range_of(gamma, lnb), range_of(beta, lnb)};
    const Range outs[] = {range_of(dQ, tok * es), range_of(dK, tok * es), range_of(dV, tok * es),
                          range_of(deta, BH * s.L * 4), range_of(dW0, ninit * dd * 4),
                          range_of(db0, ninit * s.d * 4), range_of(workspace, need),
                          range_of(dgamma, lnb), range_of(dbeta, lnb)};
    for (int o = 0; o < 9; ++o) {
        for (int o2 = o + 1; o2 < 9; ++o2)
            if (overlap(outs[o], outs[o2])) return fail(TTT_ERR_INVALID_ARG, "output buffers overlap");
        for (const Range &r : ins)
            if (overlap(outs[o], r)) return fail(TTT_ERR_INVALID_ARG, "an output overlaps an input");
    }
    const bool ln = s.residual_ln != 0;
    ttt::LinearBwdArgs a{s, Q, K, V, dZ, eta, W0, b0, ln ? gamma : nullptr, ln ? beta : nullptr, dW_final,
                         db_final, dQ, dK, dV, deta, dW0, db0, ln ? dgamma : nullptr, ln ? dbeta : nullptr,
                         workspace, reinterpret_cast<cudaStream_t>(stream)};
    cudaError_t e = ttt::launch_linear_bwd(a);
    if (e != cudaSuccess) return fail(TTT_ERR_CUDA, "ttt_linear_bwd launch: %s", cudaGetErrorString(e));
    return ok();
}

ttt_status ttt_linear_step(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                           const float *eta, float *W, float *b, const float *gamma,
                           const float *beta, void *Z, ttt_stream_t stream)
{
    ttt_status st = check_desc(desc, false);
    if (st != TTT_OK) return st;
    ttt_desc s = *desc;
    if (s.mini_batch != 1) return fail(TTT_ERR_INVALID_ARG, "ttt_linear_step needs mini_batch == 1");
    s.init_per_batch = 1;
    const void *ptrs[] = {Q, K, V, eta, W, b, Z};
    const char *names[] = {"Q", "K", "V", "eta", "W", "b", "Z"};
    for (int i = 0; i < 7; ++i)
        if ((st = check_ptr(ptrs[i], names[i])) != TTT_OK) return st;
    if (s.residual_ln) {
        if ((st = check_ptr(gamma, "gamma")) != TTT_OK) return st;
        if ((st = check_ptr(beta, "beta")) != TTT_OK) return st;
    }
    const size_t es = s.io_dtype == TTT_BF16 ? 2 : 4;
    const size_t BH = (size_t)ttt::call_rows(s), tok = BH * s.L * s.d;
    const Range rq = range_of(Q, tok * es), rk = range_of(K, tok * es), rv = range_of(V, tok * es),
                re = range_of(eta, BH * s.L * 4), rw = range_of(W, BH * s.d * s.d * 4),
                rb = range_of(b, BH * s.d * 4), rz = range_of(Z, tok * es),
                rg = range_of(gamma, s.residual_ln ? s.H * s.d * 4 : 0),
                rbe = range_of(beta, s.residual_ln ? s.H * s.d * 4 : 0);
    // the written buffers (W, b, Z) may overlap nothing; the read-only ones may share memory
    const Range written[] = {rw, rb, rz};
    const Range all[] = {rq, rk, rv, re, rw, rb, rz, rg, rbe};
    const char *wnames[] = {"W", "b", "Z"};
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 9; ++j)
            if (j != 4 + i && overlap(written[i], all[j]))
                return fail(TTT_ERR_INVALID_ARG, "%s overlaps another buffer", wnames[i]);
    ttt::LinearArgs la{s, Q, K, V, eta, W, b, gamma, beta, Z, W, b,
                       reinterpret_cast<cudaStream_t>(stream), nullptr};
    if (!ttt::linear_decode_supported(s) && !ttt::linear_generic_smem_bytes(s))
        return fail(TTT_ERR_UNSUPPORTED, "no decode kernel for d=%d", s.d);
    la.status = s.status ? s.status : failure_flag(&st);
    if (st != TTT_OK) return st;
    cudaError_t e;
    if (ttt::linear_decode_supported(s)) {
        ttt::DecodeArgs a{s, Q, K, V, eta, W, b, gamma, beta, Z, la.stream};
        e = ttt::launch_linear_decode(a);
    } else {
        e = ttt::launch_linear_generic(la);   // reads its state slice before writing it back
    }
    if (e != cudaSuccess) return fail(TTT_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return ok();
}

ttt_status ttt_mlp_fwd(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                       const float *eta, const float *W1_0, const float *b1_0,
                       const float *W2_0, const float *b2_0, const float *gamma,
                       const float *beta, void *Z, float *W1_f, float *b1_f, float *W2_f,
                       float *b2_f, ttt_stream_t stream)
{
    ttt_status st = check_desc(desc, true);
    if (st != TTT_OK) return st;
    ttt_desc s = *desc;
    if (s.d_hidden == 0) s.d_hidden = 4 * s.d;
    const void *ptrs[] = {Q, K, V, eta, W1_0, b1_0, W2_0, b2_0, Z, W1_f, b1_f, W2_f, b2_f};
    const char *names[] = {"Q", "K", "V", "eta", "W1_0", "b1_0", "W2_0", "b2_0",
                           "Z", "W1_f", "b1_f", "W2_f", "b2_f"};
    for (int i = 0; i < 13; ++i)
        if ((st = check_ptr(ptrs[i], names[i])) != TTT_OK) return st;
    if (s.residual_ln) {
        if ((st = check_ptr(gamma, "gamma")) != TTT_OK) return st;
        if ((st = check_ptr(beta, "beta")) != TTT_OK) return st;
    }
    const size_t es = s.io_dtype == TTT_BF16 ? 2 : 4;
    const size_t BH = (size_t)ttt::call_rows(s), ninit = s.init_per_batch ? BH : (size_t)s.H;
    const size_t n1 = (size_t)s.d * s.d_hidden;
    const size_t seq = BH * s.L * s.d;
    Range ins[] = {range_of(Q, seq * es), range_of(K, seq * es), range_of(V, seq * es),
                   range_of(eta, BH * s.L * 4), range_of(W1_0, ninit * n1 * 4),
                   range_of(b1_0, ninit * s.d_hidden * 4), range_of(W2_0, ninit * n1 * 4),
                   range_of(b2_0, ninit * s.d * 4),
                   range_of(gamma, s.residual_ln ? s.H * s.d * 4 : 0),
                   range_of(beta, s.residual_ln ? s.H * s.d * 4 : 0)};
    Range outs[] = {range_of(Z, seq * es), range_of(W1_f, BH * n1 * 4),
                    range_of(b1_f, BH * s.d_hidden * 4), range_of(W2_f, BH * n1 * 4),
                    range_of(b2_f, BH * s.d * 4)};
    for (int o = 0; o < 5; ++o) {
        for (int o2 = o + 1; o2 < 5; ++o2)
            if (overlap(outs[o], outs[o2])) return fail(TTT_ERR_INVALID_ARG, "output buffers overlap");
        for (int i = 0; i < 10; ++i) {
            // final state o (1..4) may sit exactly on initial state i = o + 3 when per batch
            bool same = s.init_per_batch && o >= 1 && i == o + 3 && outs[o].lo == ins[i].lo;
            if (overlap(outs[o], ins[i]) && !same)
                return fail(TTT_ERR_INVALID_ARG, "%s overlaps an input", names[8 + o]);
        }
    }
    const char *kname = mlp_kernel(s);
    if (!kname)
        return fail(TTT_ERR_UNSUPPORTED, "no kernel for d=%d d_hidden=%d mini_batch=%d", s.d,
                    s.d_hidden, s.mini_batch);
    ttt::MlpArgs a{s, Q, K, V, eta, W1_0, b1_0, W2_0, b2_0, gamma, beta, Z,
                   W1_f, b1_f, W2_f, b2_f, reinterpret_cast<cudaStream_t>(stream), nullptr};
    a.status = s.status ? s.status : failure_flag(&st);
    if (st != TTT_OK) return st;
    cudaError_t e = kname == kMlpTmem    ? ttt::launch_mlp_tmem(a)
                    : kname == kMlpFused ? ttt::launch_mlp_tc(a)
                                         : ttt::launch_mlp_generic(a);
    if (e != cudaSuccess) return fail(TTT_ERR_CUDA, "%s launch: %s", kname, cudaGetErrorString(e));
    return ok();
}

ttt_status ttt_eta_gate(int B, int H, int L, int d_model, ttt_dtype x_dtype, float eta_base,
                        const void *x, const float *theta, float *eta, int max_sms, ttt_stream_t stream)
{
    if (B <= 0 || H <= 0 || L <= 0 || d_model <= 0)
        return fail(TTT_ERR_INVALID_ARG, "B, H, L and d_model must be positive");
    if (max_sms < 0) return fail(TTT_ERR_INVALID_ARG, "max_sms must be >= 0");
    if (x_dtype != TTT_F32 && x_dtype != TTT_BF16)
        return fail(TTT_ERR_INVALID_ARG, "x_dtype must be TTT_F32 or TTT_BF16");
    if (!std::isfinite(eta_base)) return fail(TTT_ERR_INVALID_ARG, "eta_base must be finite");
    if ((long long)B * L > 0x7fffffffLL || (long long)B * H * L > (1LL << 40))
        return fail(TTT_ERR_INVALID_ARG, "B * L exceeds the supported size");
    if (x_dtype == TTT_BF16 && d_model % 8 != 0)
        return fail(TTT_ERR_INVALID_ARG, "d_model must be a multiple of 8 for bf16 tokens");
    ttt_status st;
    if ((st = check_ptr(x, "x")) != TTT_OK) return st;
    if ((st = check_ptr(theta, "theta")) != TTT_OK) return st;
    if ((st = check_ptr(eta, "eta")) != TTT_OK) return st;
    const size_t es = x_dtype == TTT_BF16 ? 2 : 4;
    const Range re = range_of(eta, (size_t)B * H * L * 4);
    if (overlap(re, range_of(x, (size_t)B * L * d_model * es)) ||
        overlap(re, range_of(theta, (size_t)H * d_model * 4)))
        return fail(TTT_ERR_INVALID_ARG, "eta overlaps an input");
    ttt::GateArgs a{B, H, L, d_model, x_dtype, eta_base, x, theta, eta,
                    reinterpret_cast<cudaStream_t>(stream), nullptr, max_sms};
    a.status = failure_flag(&st);
    if (st != TTT_OK) return st;
    cudaError_t e = ttt::launch_eta_gate(a);
    if (e != cudaSuccess) return fail(TTT_ERR_CUDA, "eta gate launch: %s", cudaGetErrorString(e));
    return ok();
}

ttt_status ttt_qkv_proj(int B, int H, int L, int d_model, int d, const void *x, const void *W, void *Q,
                        void *K, void *V, int max_sms, ttt_stream_t stream)
{
    if (B <= 0 || H <= 0 || L <= 0 || d_model <= 0 || d <= 0)
        return fail(TTT_ERR_INVALID_ARG, "B, H, L, d_model and d must be positive");
    if (max_sms < 0) return fail(TTT_ERR_INVALID_ARG, "max_sms must be >= 0");
    if ((long long)B * L > 0x7fffffffLL || 3LL * H * d > 0x7fffffffLL || (long long)B * H * L * d > (1LL << 40))
        return fail(TTT_ERR_INVALID_ARG, "the sizes exceed the supported range");
    ttt_status st;
    const void *ptrs[] = {x, W, Q, K, V};
    const char *names[] = {"x", "W", "Q", "K", "V"};
    for (int i = 0; i < 5; ++i)
        if ((st = check_ptr(ptrs[i], names[i])) != TTT_OK) return st;
    if (!ttt::qkv_proj_supported(B, H, L, d_model, d))
        return fail(TTT_ERR_UNSUPPORTED, "the projection kernel takes d = 64, d_model a multiple of 64 and "
                                         "3 H d a multiple of 256 (B=%d H=%d d_model=%d d=%d)", B, H, d_model, d);
    const size_t nx = (size_t)B * L * d_model * 2, nw = (size_t)3 * H * d * d_model * 2, no = (size_t)B * H * L * d * 2;
    const Range outs[] = {range_of(Q, no), range_of(K, no), range_of(V, no)};
    const Range ins[] = {range_of(x, nx), range_of(W, nw)};
    for (int o = 0; o < 3; ++o) {
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlap(outs[o], outs[o2])) return fail(TTT_ERR_INVALID_ARG, "Q, K, V overlap");
        for (const Range &r : ins)
            if (overlap(outs[o], r)) return fail(TTT_ERR_INVALID_ARG, "an output overlaps an input");
    }
    ttt::ProjArgs a{B, H, L, d_model, d, x, W, static_cast<__nv_bfloat16 *>(Q), static_cast<__nv_bfloat16 *>(K),
                    static_cast<__nv_bfloat16 *>(V), reinterpret_cast<cudaStream_t>(stream), nullptr, max_sms};
    a.status = failure_flag(&st);
    if (st != TTT_OK) return st;
    cudaError_t e = ttt::launch_qkv_proj(a);
    if (e != cudaSuccess) return fail(TTT_ERR_CUDA, "projection launch: %s", cudaGetErrorString(e));
    return ok();
}

void ttt_set_wait_timeout_ns(long long ns) { ttt::set_wait_timeout_ns(ns); }

void ttt_debug_withhold_loads(int on) { ttt::set_withhold_loads(on); }

ttt_status ttt_sync_status(ttt_stream_t stream)
{
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return fail(TTT_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    // the flag read is the one of the stream's device (the legacy default stream belongs to
    // the current device); the current device is restored afterwards
    int cur = 0, dev = 0;
    if ((e = cudaGetDevice(&cur)) != cudaSuccess)
        return fail(TTT_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    dev = cur;
    if (cs != nullptr && (e = cudaStreamGetDevice(cs, &dev)) != cudaSuccess)
        return fail(TTT_ERR_CUDA, "cudaStreamGetDevice: %s", cudaGetErrorString(e));
    if (dev != cur && (e = cudaSetDevice(dev)) != cudaSuccess)
        return fail(TTT_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(e));
    unsigned int flag = 0;
    cudaError_t e_clear = cudaSuccess;
    e = cudaMemcpyFromSymbol(&flag, g_ttt_failure_flag, sizeof(flag));
    if (e == cudaSuccess && flag != ttt::kStatusOk) {
        const unsigned int zero = 0;
        e_clear = cudaMemcpyToSymbol(g_ttt_failure_flag, &zero, sizeof(zero));
    }
    if (dev != cur) cudaSetDevice(cur);
    if (e != cudaSuccess) return fail(TTT_ERR_CUDA, "reading the failure flag: %s", cudaGetErrorString(e));
    if (e_clear != cudaSuccess)
        return fail(TTT_ERR_CUDA, "clearing the failure flag (0x%x): %s", flag, cudaGetErrorString(e_clear));
    if (flag != ttt::kStatusOk)
        return fail(TTT_ERR_TIMEOUT, "a kernel gave up on a bounded wait (flag 0x%x)", flag);
    return ok();
}

}  // extern "C"
