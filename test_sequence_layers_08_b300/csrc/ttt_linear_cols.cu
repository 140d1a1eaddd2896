// ttt_linear_cols.cu -- TTT-Linear without the residual LayerNorm, one (batch, head) scan
// split over several CTAs by output column.
//
// Without the output LayerNorm the inner loop of the damodev.csdn.net TTT article
// (sections 4.1-4.2; f(k) = k W + c, squared-error or inner-product loss, optional weight
// decay of the ai-feeds Modular TTT page) never mixes the columns of the state: column j of
// W and c evolves from column j of K W + c, of V and of G alone,
//   G[:, j] = (K W + 1 c)[:, j] - V[:, j]          (inner product: -V[:, j])
//   Z[:, j] = f . (Q W)[:, j] + c_j - (tril(Q K^T + 1) diag(eta)) G[:, j]
//   W[:, j] <- (1 - lambda sum eta) W[:, j] - K^T diag(eta) G[:, j],  c_j -= eta^T G[:, j]
// (f_t = 1 - lambda sum_{s<=t} eta_s).  Only the mini-batch Gram Q K^T is shared by all
// columns, and it depends on the inputs alone.  So a (batch, head) row is split over S CTAs
// that each own DC consecutive columns and need no communication: each reads the whole
// Q, K tiles and its columns of V, W0, b0, recomputes the Gram, and writes its columns of
// Z, W_final, b_final.  A row that would use one SM now uses S, and each step's latency
// shrinks with the columns: the d-long contractions are further split over threads and
// reduced through shared memory.
//
// B300 design (fp32 FFMA, 256 threads; for workloads with few (batch, head) rows, where the
// one-CTA-per-row kernels leave most of the 148 SMs idle):
//   * Q and K rows are stored with a 4-float pad (row stride d + 4): threads that read the
//     same column of different tokens hit different shared-memory banks; W rows are read as
//     broadcasts (threads of a group share the contraction slice);
//   * tiles are double-buffered, so a step needs three block barriers: after staging,
//     after the products and the Gram, after G;
//   * the next mini-batch's Q, K, V columns and eta are loaded into registers while the
//     current one computes (when they fit in four 16-byte vectors per thread).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr int kPrefetchVec = 4;
constexpr size_t kMaxSmem = 227 * 1024;

struct ColsParams {
    int H, L, d, mb, init_per_batch, ip, S, US;
    float wd;
    const void *Q, *K, *V;
    const float *eta, *W0, *b0;
    void *Z;
    float *Wf, *bf;
    int hoff;
};

template <typename IO> struct Io4;
template <> struct Io4<float> {
    using T = float4;
    static __device__ __forceinline__ float4 load(const float *p, size_t i)
    {
        return *reinterpret_cast<const float4 *>(p + i);
    }
    static __device__ __forceinline__ float4 f32(float4 v) { return v; }
    static __device__ __forceinline__ void store(float *p, size_t i, float4 v)
    {
        p[i] = v.x;
        p[i + 1] = v.y;
        p[i + 2] = v.z;
        p[i + 3] = v.w;
    }
};
template <> struct Io4<__nv_bfloat16> {
    using T = uint2;
    static __device__ __forceinline__ uint2 load(const __nv_bfloat16 *p, size_t i)
    {
        return *reinterpret_cast<const uint2 *>(p + i);
    }
    static __device__ __forceinline__ float4 f32(uint2 v)
    {
        return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, size_t i, float4 v)
    {
        p[i] = __float2bfloat16_rn(v.x);
        p[i + 1] = __float2bfloat16_rn(v.y);
        p[i + 2] = __float2bfloat16_rn(v.z);
        p[i + 3] = __float2bfloat16_rn(v.w);
    }
};

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void fma4(float4 &a, float s, float4 b)
{
    a.x = fmaf(s, b.x, a.x);
    a.y = fmaf(s, b.y, a.y);
    a.z = fmaf(s, b.z, a.z);
    a.w = fmaf(s, b.w, a.w);
}
__device__ __forceinline__ void add4(float4 &a, float4 b)
{
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// Shared-memory plan (floats), shared by the kernel and the host's size check.
struct ColsLayout {
    int ds;                        // padded Q/K row stride
    int W, c, K, Q, V, et, G, Zb, At, Pk, Pq, total;
    __host__ __device__ ColsLayout(int d, int mb, int dc, int us)
    {
        ds = d + 4;
        W = 0;
        c = W + d * dc;
        K = c + ((dc + 3) & ~3);
        Q = K + 2 * mb * ds;       // two buffers each
        V = Q + 2 * mb * ds;
        et = V + 2 * mb * dc;
        G = et + 2 * ((mb + 3) & ~3);
        Zb = G + mb * dc;
        At = Zb + mb * dc;
        Pk = At + ((mb * mb + 3) & ~3);
        Pq = Pk + us * mb * dc;
        total = Pq + us * mb * dc;
    }
};

// Contraction split: the largest power of two US (US <= d / 4, d / US a multiple of 4) with
// the partial products and the Gram fitting one pass of the block's threads.
__host__ __device__ constexpr int cols_us(int d, int mb, int dc)
{
    int us = 1;
    while (2 * us <= d / 4 && (d / (2 * us)) % 4 == 0 && 2 * us * (dc / 4) * mb + mb * (mb + 1) / 2 <= kThreads)
        us *= 2;
    return us;
}

// DT, MT: the head dim and the mini-batch size as compile-time constants (0: taken from the
// parameters at run time).  With both fixed, the item decodes are shifts and the d- and
// b-long loops unroll, so their shared-memory loads are issued back to back.
template <typename IO, int DC, int DT, int MT>
__global__ void __launch_bounds__(kThreads) linear_cols_kernel(ColsParams p)
{
    constexpr int DC4 = DC / 4;
    constexpr int UST = (DT && MT) ? cols_us(DT, MT, DC) : 0;
    extern __shared__ float4 sm4[];
    float *sm = reinterpret_cast<float *>(sm4);
    const int d = DT ? DT : p.d, mb = MT ? MT : p.mb, L = p.L, US = UST ? UST : p.US, ul = d / US;
    const ColsLayout lay(d, mb, DC, US);
    const int ds = lay.ds;
    float *W = sm + lay.W, *c = sm + lay.c, *G = sm + lay.G, *Zb = sm + lay.Zb, *At = sm + lay.At;
    float4 *Pk = reinterpret_cast<float4 *>(sm + lay.Pk), *Pq = reinterpret_cast<float4 *>(sm + lay.Pq);
    const int row = blockIdx.x / p.S, part = blockIdx.x - row * p.S, j0 = part * DC;
    const int h = (p.hoff + row) % p.H, tid = threadIdx.x;

    const size_t init = p.init_per_batch ? (size_t)row : (size_t)h;
    for (int i = tid; i < d * DC; i += kThreads) {
        const int u = i / DC, jl = i - u * DC;
        W[i] = p.W0[(init * d + u) * d + j0 + jl];
    }
    for (int jl = tid; jl < DC; jl += kThreads) c[jl] = p.b0[init * d + j0 + jl];

    const IO *Qg = static_cast<const IO *>(p.Q) + (size_t)row * L * d;
    const IO *Kg = static_cast<const IO *>(p.K) + (size_t)row * L * d;
    const IO *Vg = static_cast<const IO *>(p.V) + (size_t)row * L * d;
    IO *Zg = static_cast<IO *>(p.Z) + (size_t)row * L * d;
    const float *eg = p.eta + (size_t)row * L;

    // the vectors of one mini-batch: K rows, Q rows (d / 4 each per token), then this CTA's
    // V columns (DC / 4 per token)
    const int nk4 = mb * (d >> 2), nv4 = mb * DC4, nvec = 2 * nk4 + nv4;
    const bool prefetch = nvec <= kPrefetchVec * kThreads;
    using V4 = Io4<IO>;
    typename V4::T pre[kPrefetchVec];
    float pre_eta = 0.f;
    auto src_of = [&](int v, int n0, int &which, int &t, int &col) {
        if (v < 2 * nk4) {
            which = v < nk4 ? 0 : 1;
            const int i = v - which * nk4;
            t = i / (d >> 2);
            col = (i - t * (d >> 2)) * 4;
            return (size_t)(n0 + t) * d + col;
        }
        which = 2;
        const int i = v - 2 * nk4;
        t = i / DC4;
        col = (i - t * DC4) * 4;
        return (size_t)(n0 + t) * d + j0 + col;
    };
    auto fetch = [&](int n0) {
        if (tid < mb) pre_eta = eg[n0 + tid];
#pragma unroll
        for (int r = 0; r < kPrefetchVec; ++r) {
            const int v = tid + r * kThreads;
            if (v < nvec) {
                int which, t, col;
                const size_t o = src_of(v, n0, which, t, col);
                pre[r] = V4::load(which == 0 ? Kg : which == 1 ? Qg : Vg, o);
            }
        }
    };
    auto put = [&](int buf, int which, int t, int col, float4 x) {
        float *dst = which == 0   ? sm + lay.K + buf * mb * ds + t * ds + col
                     : which == 1 ? sm + lay.Q + buf * mb * ds + t * ds + col
                                  : sm + lay.V + buf * mb * DC + t * DC + col;
        st4(dst, x);
    };
    auto stage = [&](int n0, int buf) {
        float *et = sm + lay.et + buf * ((mb + 3) & ~3);
        if (prefetch) {
#pragma unroll
            for (int r = 0; r < kPrefetchVec; ++r) {
                const int v = tid + r * kThreads;
                if (v < nvec) {
                    int which, t, col;
                    src_of(v, n0, which, t, col);
                    put(buf, which, t, col, V4::f32(pre[r]));
                }
            }
            if (tid < mb) et[tid] = pre_eta;
        } else {
            for (int v = tid; v < nvec; v += kThreads) {
                int which, t, col;
                const size_t o = src_of(v, n0, which, t, col);
                put(buf, which, t, col, V4::f32(V4::load(which == 0 ? Kg : which == 1 ? Qg : Vg, o)));
            }
            for (int s = tid; s < mb; s += kThreads) et[s] = eg[n0 + s];
        }
    };

    const int nprod = US * DC4 * mb, ngram = mb * (mb + 1) / 2;
    if (prefetch) fetch(0);
    for (int n0 = 0, n = 0; n0 < L; n0 += mb, ++n) {
        const int buf = n & 1;
        stage(n0, buf);
        __syncthreads();   // tiles staged; the previous step's W, c updates visible
        if (prefetch && n0 + mb < L) fetch(n0 + mb);
        const float *Kt = sm + lay.K + buf * mb * ds, *Qt = sm + lay.Q + buf * mb * ds;
        const float *Vt = sm + lay.V + buf * mb * DC, *et = sm + lay.et + buf * ((mb + 3) & ~3);

        // (A) partial products over a slice of the contraction: item (us, j4, t), t fastest
        //     (the group shares the W rows: broadcasts); and the Gram
        //     At[s][t] = eta_s (q_t . k_s + 1), s <= t
        for (int i = tid; i < nprod + ngram; i += kThreads) {
            if (i < nprod) {
                const int t = i % mb, r = i / mb, j4 = r % DC4, us = r / DC4;
                const float *kr = Kt + t * ds, *qr = Qt + t * ds;
                const float *wr = W + j4 * 4;
                float4 ak = make_float4(0.f, 0.f, 0.f, 0.f), aq = ak;
                const int u0 = us * ul;
#pragma unroll
                for (int u = u0; u < u0 + ul; u += 4) {
                    const float4 k4 = ld4(kr + u), q4 = ld4(qr + u);
                    const float4 w0 = ld4(wr + u * DC), w1 = ld4(wr + (u + 1) * DC);
                    const float4 w2 = ld4(wr + (u + 2) * DC), w3 = ld4(wr + (u + 3) * DC);
                    if (!p.ip) {
                        fma4(ak, k4.x, w0); fma4(ak, k4.y, w1); fma4(ak, k4.z, w2); fma4(ak, k4.w, w3);
                    }
                    fma4(aq, q4.x, w0); fma4(aq, q4.y, w1); fma4(aq, q4.z, w2); fma4(aq, q4.w, w3);
                }
                Pk[(us * DC4 + j4) * mb + t] = ak;
                Pq[(us * DC4 + j4) * mb + t] = aq;
            } else {
                const int g = i - nprod;
                int t = (int)((sqrtf(8.f * g + 1.f) - 1.f) * 0.5f);
                while ((t + 1) * (t + 2) / 2 <= g) ++t;
                while (t * (t + 1) / 2 > g) --t;
                const int s = g - t * (t + 1) / 2;
                const float *qr = Qt + t * ds, *kr = Kt + s * ds;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int u = 0; u < d; u += 4) {
                    const float4 q4 = ld4(qr + u), k4 = ld4(kr + u);
                    a0 = fmaf(q4.x, k4.x, a0);
                    a1 = fmaf(q4.y, k4.y, a1);
                    a0 = fmaf(q4.z, k4.z, a0);
                    a1 = fmaf(q4.w, k4.w, a1);
                }
                At[s * mb + t] = (a0 + a1 + 1.f) * et[s];
            }
        }
        __syncthreads();

        // (B) reduce the partials: G (key side) and the query side at the starting weights
        for (int i = tid; i < mb * DC4; i += kThreads) {
            const int t = i % mb, j4 = i / mb;
            float4 ak = ld4(c + j4 * 4), aq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int us = 0; us < US; ++us) {
                if (!p.ip) add4(ak, Pk[(us * DC4 + j4) * mb + t]);
                add4(aq, Pq[(us * DC4 + j4) * mb + t]);
            }
            const float4 v4 = ld4(Vt + t * DC + j4 * 4);
            const float4 g4 = p.ip ? make_float4(-v4.x, -v4.y, -v4.z, -v4.w)
                                   : make_float4(ak.x - v4.x, ak.y - v4.y, ak.z - v4.z, ak.w - v4.w);
            st4(G + t * DC + j4 * 4, g4);
            float f = 1.f;
            if (p.wd != 0.f) {
                float cum = 0.f;
                for (int s = 0; s <= t; ++s) cum += et[s];
                f = 1.f - p.wd * cum;
            }
            const float4 c4 = ld4(c + j4 * 4);
            st4(Zb + t * DC + j4 * 4, make_float4(fmaf(f, aq.x, c4.x), fmaf(f, aq.y, c4.y), fmaf(f, aq.z, c4.z),
                                                  fmaf(f, aq.w, c4.w)));
        }
        __syncthreads();

        // (C) outputs Z[t] = Zb[t] - sum_{s <= t} At[s][t] G[s]; the state update
        //     W[u] <- decay W[u] - sum_s eta_s K[s][u] G[s]; c -= eta^T G
        float decay = 1.f;
        if (p.wd != 0.f) {
            float tot = 0.f;
            for (int s = 0; s < mb; ++s) tot += et[s];
            decay = 1.f - p.wd * tot;
        }
        const int nout = mb * DC4, nupd = d * DC4;
        for (int i = tid; i < nout + nupd + DC; i += kThreads) {
            if (i < nout) {
                const int j4 = i % DC4, t = i / DC4;
                float4 z = ld4(Zb + t * DC + j4 * 4);
#pragma unroll
                for (int s = 0; s < mb; ++s)
                    if (s <= t) fma4(z, -At[s * mb + t], ld4(G + s * DC + j4 * 4));
                V4::store(Zg, (size_t)(n0 + t) * d + j0 + j4 * 4, z);
            } else if (i < nout + nupd) {
                const int k = i - nout, j4 = k % DC4, u = k / DC4;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int s = 0; s < mb; ++s) fma4(a, et[s] * Kt[s * ds + u], ld4(G + s * DC + j4 * 4));
                float *w = W + u * DC + j4 * 4;
                const float4 w4 = ld4(w);
                st4(w, make_float4(fmaf(decay, w4.x, -a.x), fmaf(decay, w4.y, -a.y), fmaf(decay, w4.z, -a.z),
                                   fmaf(decay, w4.w, -a.w)));
            } else {
                const int jl = i - nout - nupd;
                float a = 0.f;
#pragma unroll
                for (int s = 0; s < mb; ++s) a = fmaf(et[s], G[s * DC + jl], a);
                c[jl] -= a;
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < d * DC; i += kThreads) {
        const int u = i / DC, jl = i - u * DC;
        p.Wf[((size_t)row * d + u) * d + j0 + jl] = W[i];
    }
    for (int jl = tid; jl < DC; jl += kThreads) p.bf[(size_t)row * d + j0 + jl] = c[jl];
}

}  // namespace

int linear_cols_dc(const ttt_desc &s)
{
    if (s.residual_ln || s.d > 128 || s.d % 4 != 0 || s.mini_batch > 64) return 0;
    const int rows = call_rows(s);
    // columns per CTA: the fewest (down to 4) that keep the grid within two CTAs per SM
    constexpr int kSmCtas = 2 * 148;
    for (int dc : {4, 8, 16}) {
        if (s.d % dc != 0 || s.d / dc < 2) continue;
        if ((long long)rows * (s.d / dc) > kSmCtas) continue;
        const ColsLayout lay(s.d, s.mini_batch, dc, cols_us(s.d, s.mini_batch, dc));
        if ((size_t)lay.total * sizeof(float) > kMaxSmem) continue;
        return dc;
    }
    return 0;
}

cudaError_t launch_linear_cols(const LinearArgs &a)
{
    const ttt_desc &s = a.desc;
    const int dc = linear_cols_dc(s);
    if (!dc) return cudaErrorInvalidValue;
    const int us = cols_us(s.d, s.mini_batch, dc);
    ColsParams p{s.H, s.L, s.d, s.mini_batch, s.init_per_batch, s.loss == TTT_LOSS_INNER_PRODUCT, s.d / dc, us,
                 s.weight_decay, a.Q, a.K, a.V, a.eta, a.W0, a.b0, a.Z, a.W_final, a.b_final, head_offset(s)};
    const size_t smem = (size_t)ColsLayout(s.d, s.mini_batch, dc, us).total * sizeof(float);
    const bool f32 = s.io_dtype == TTT_F32, fixed = s.d == 64 && s.mini_batch == 16;
    auto pick = [&](auto kf, auto kf_any, auto kb, auto kb_any) {
        return f32 ? (fixed ? (const void *)kf : (const void *)kf_any) : (fixed ? (const void *)kb : (const void *)kb_any);
    };
    const void *k = nullptr;
    switch (dc) {
    case 4:
        k = pick(linear_cols_kernel<float, 4, 64, 16>, linear_cols_kernel<float, 4, 0, 0>,
                 linear_cols_kernel<__nv_bfloat16, 4, 64, 16>, linear_cols_kernel<__nv_bfloat16, 4, 0, 0>);
        break;
    case 8:
        k = pick(linear_cols_kernel<float, 8, 64, 16>, linear_cols_kernel<float, 8, 0, 0>,
                 linear_cols_kernel<__nv_bfloat16, 8, 64, 16>, linear_cols_kernel<__nv_bfloat16, 8, 0, 0>);
        break;
    default:
        k = pick(linear_cols_kernel<float, 16, 64, 16>, linear_cols_kernel<float, 16, 0, 0>,
                 linear_cols_kernel<__nv_bfloat16, 16, 64, 16>, linear_cols_kernel<__nv_bfloat16, 16, 0, 0>);
        break;
    }
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {&p};
    return cudaLaunchKernel(k, dim3(call_rows(s) * p.S), dim3(kThreads), args, smem, a.stream);
}

}  // namespace ttt
