// ttt_generic.cu -- generic TTT inner-loop forward kernels (any small shape).
//
// One CTA per (batch, head) scans the L / b mini-batches in order.  The fast
// weights live in shared memory in fp32 for the whole scan; every contraction
// is plain fp32 FFMA.  These kernels serve fp32 I/O (where a relative error of
// 1e-5 rules out tf32/bf16 tensor-core operands) with the residual LayerNorm or
// with many (batch, head) rows (without LayerNorm and with few rows the
// column-split kernel takes it), the TTT-MLP in fp32, and every shape the
// tensor-core kernels do not take.
//
// Per mini-batch (damodev.csdn.net TTT article, sections 4.1-4.2; lryc.cn TTT
// article, section 2.1 for the MLP and the residual LayerNorm):
//   Zk = K W + 1c,  G = dl/dZk  (Zk - V, or the LayerNorm-fused L2 backward
//                                against V - K),
//   A  = tril(Q K^T + 1) diag(eta)           (diagonal included),
//   Zb = Q W + 1c - A G,  out = Zb or Q + LN(Zb),
//   W -= K^T diag(eta) G,  c -= eta^T G.
// The MLP does the same per layer, with X2 = GELU(Z1) as the second layer's
// input and the back-propagated G1 = (G2 W2^T) * GELU'(Z1).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float load_io(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_io(const __nv_bfloat16 *p, size_t i)
{
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_io(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_io(__nv_bfloat16 *p, size_t i, float v)
{
    p[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Mean and 1/sqrt(biased var + eps) of one row, two passes; whole warp.
__device__ __forceinline__ void row_stats(const float *z, int d, float eps, float &mu,
                                          float &r)
{
    const int lane = threadIdx.x & 31;
    float s = 0.f;
    for (int j = lane; j < d; j += 32) s += z[j];
    mu = warp_sum(s) / d;
    float v = 0.f;
    for (int j = lane; j < d; j += 32) {
        float t = z[j] - mu;
        v += t * t;
    }
    r = rsqrtf(warp_sum(v) / d + eps);
}

// In place: z <- d/dz 1/2 || gamma * norm(z) + beta - y ||^2, y = v - k.
__device__ void ln_l2_bwd_row(float *z, const float *v, const float *k, const float *gam,
                              const float *bet, int d, float eps)
{
    const int lane = threadIdx.x & 31;
    float mu, r;
    row_stats(z, d, eps, mu, r);
    float m1 = 0.f, m2 = 0.f;
    for (int j = lane; j < d; j += 32) {
        float xh = (z[j] - mu) * r;
        float gx = gam[j] * (gam[j] * xh + bet[j] - (v[j] - k[j]));
        m1 += gx;
        m2 += gx * xh;
    }
    m1 = warp_sum(m1) / d;
    m2 = warp_sum(m2) / d;
    __syncwarp();
    for (int j = lane; j < d; j += 32) {
        float xh = (z[j] - mu) * r;
        float gx = gam[j] * (gam[j] * xh + bet[j] - (v[j] - k[j]));
        z[j] = r * (gx - m1 - xh * m2);
    }
    __syncwarp();
}

// In place: z <- d/dz of -< q + gamma * norm(z) + beta, v > (inner-product loss).
__device__ void ln_ip_bwd_row(float *z, const float *v, const float *gam, int d, float eps)
{
    const int lane = threadIdx.x & 31;
    float mu, r;
    row_stats(z, d, eps, mu, r);
    float m1 = 0.f, m2 = 0.f;
    for (int j = lane; j < d; j += 32) {
        float xh = (z[j] - mu) * r;
        float gx = -gam[j] * v[j];
        m1 += gx;
        m2 += gx * xh;
    }
    m1 = warp_sum(m1) / d;
    m2 = warp_sum(m2) / d;
    __syncwarp();
    for (int j = lane; j < d; j += 32) {
        float xh = (z[j] - mu) * r;
        z[j] = r * (-gam[j] * v[j] - m1 - xh * m2);
    }
    __syncwarp();
}

// Sum of eta over tokens 0..t of the staged mini-batch.
__device__ __forceinline__ float eta_prefix(const float *et, int t)
{
    float a = 0.f;
    for (int s = 0; s <= t; ++s) a += et[s];
    return a;
}

// out_row = q + gamma * norm(z) + beta, written to global in the I/O type.
template <typename IO>
__device__ void ln_out_row(const float *z, const float *q, const float *gam,
                           const float *bet, int d, float eps, IO *out)
{
    const int lane = threadIdx.x & 31;
    float mu, r;
    row_stats(z, d, eps, mu, r);
    for (int j = lane; j < d; j += 32) store_io(out, j, q[j] + gam[j] * (z[j] - mu) * r + bet[j]);
}

__device__ __forceinline__ float gelu_tanh(float x)
{
    const float s = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * x * (1.f + tanhf(s * (x + 0.044715f * x * x * x)));
}

__device__ __forceinline__ float gelu_tanh_prime(float x)
{
    const float s = 0.7978845608028654f;
    float th = tanhf(s * (x + 0.044715f * x * x * x));
    return 0.5f * (1.f + th) + 0.5f * x * (1.f - th * th) * s * (1.f + 3.f * 0.044715f * x * x);
}

// Subtract the mean of the n values v[0..n) (shared memory, just written by the block) from
// each of them; returns the mean.  Every thread sums in the same order, so all agree on it.
__device__ float shift_by_mean(float *v, int n)
{
    __syncthreads();
    float s = 0.f;
    for (int j = 0; j < n; ++j) s += v[j];
    const float mean = s / n;
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += blockDim.x) v[j] -= mean;
    return mean;
}

struct LinearParams {
    int H, L, d, mb, ln, init_per_batch;
    float eps;
    int ip;                  // inner-product loss
    float wd;                // weight decay lambda
    const void *Q, *K, *V;
    const float *eta, *W0, *b0, *gamma, *beta;
    void *Z;
    float *Wf, *bf;
    int hoff = 0;            // head index of row 0 of this call
};

// ---------------------------------------------------------------------------
// TTT-Linear
//
// The d x d products are register-tiled: a thread owns 4 consecutive features (a float4 of
// a W row) of one token, or a 4 x 4 block of W for the update, and reads its operands as
// 16-byte shared-memory loads.  When the next mini-batch's K, Q, V fit in four 16-byte
// registers per thread, they are loaded from global memory while the current one computes.
// d must be a multiple of 4 (checked at launch).
// ---------------------------------------------------------------------------
constexpr int kLinThreads = 256;  // threads of the TTT-Linear kernel
constexpr int kLinWarps = kLinThreads / 32;
constexpr int kPrefetchVec = 4;   // 16-byte vectors of K, Q, V a thread may hold in registers

template <typename IO> struct Vec4;
template <> struct Vec4<float> {
    using T = float4;
    static __device__ __forceinline__ float4 load(const float *p, size_t i)
    {
        return *reinterpret_cast<const float4 *>(p + i);
    }
    static __device__ __forceinline__ float4 to_f32(float4 v) { return v; }
};
template <> struct Vec4<__nv_bfloat16> {
    using T = uint2;
    static __device__ __forceinline__ uint2 load(const __nv_bfloat16 *p, size_t i)
    {
        return *reinterpret_cast<const uint2 *>(p + i);
    }
    static __device__ __forceinline__ float4 to_f32(uint2 v)
    {
        return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    }
};

__device__ __forceinline__ float4 f4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void fma4(float4 &a, float s, float4 b)
{
    a.x = fmaf(s, b.x, a.x);
    a.y = fmaf(s, b.y, a.y);
    a.z = fmaf(s, b.z, a.z);
    a.w = fmaf(s, b.w, a.w);
}

// DC: the head dim as a compile-time constant (0: taken from the parameters at run time)
template <typename IO, bool LN, int DC>
__global__ void __launch_bounds__(kLinThreads) linear_generic_kernel(LinearParams p)
{
    constexpr int kThreads = kLinThreads, kWarps = kLinWarps;
    extern __shared__ float4 sm4[];
    float *sm = reinterpret_cast<float *>(sm4);
    const int d = DC ? DC : p.d, mb = p.mb, L = p.L;
    const int bh = blockIdx.x, h = (p.hoff + bh) % p.H;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int d4 = d >> 2;
    float *W = sm;                 // d*d
    float *c = W + d * d;          // d
    float *Kt = c + d;             // mb*d
    float *Qt = Kt + mb * d;
    float *Vt = Qt + mb * d;
    float *G = Vt + mb * d;        // Zk, then G
    float *Zb = G + mb * d;
    float *A = Zb + mb * d;        // mb*mb
    float *et = A + mb * mb;       // mb
    float *gam = et + mb;          // d
    float *bet = gam + d;          // d

    const size_t init = p.init_per_batch ? (size_t)bh : (size_t)h;
    for (int i = tid; i < d * d; i += kThreads) W[i] = p.W0[init * d * d + i];
    for (int j = tid; j < d; j += kThreads) {
        c[j] = p.b0[init * d + j];
        if (LN) {
            gam[j] = p.gamma[(size_t)h * d + j];
            bet[j] = p.beta[(size_t)h * d + j];
        }
    }
    // LayerNorm pivot: LN and its backward do not see a common shift of k W + c, so with the
    // residual LayerNorm the scan runs on c - mean(b0) and the mean is added back to b_final.
    // The shifted bias keeps its per-feature deviations at full fp32 precision when b0 has a
    // large common offset (an unshifted fp32 c holds them only to ulp(|c|)).
    const float pivot = LN ? shift_by_mean(c, d) : 0.f;
    const IO *Qg = static_cast<const IO *>(p.Q) + (size_t)bh * L * d;
    const IO *Kg = static_cast<const IO *>(p.K) + (size_t)bh * L * d;
    const IO *Vg = static_cast<const IO *>(p.V) + (size_t)bh * L * d;
    IO *Zg = static_cast<IO *>(p.Z) + (size_t)bh * L * d;
    const float *eg = p.eta + (size_t)bh * L;
    const int nt = mb * d, nt4 = nt >> 2;

    // K, Q, V of a mini-batch: 3 nt4 vectors of 4 elements; vector v of the three tiles
    const bool prefetch = 3 * nt4 <= kPrefetchVec * kThreads;
    using V4 = Vec4<IO>;
    typename V4::T pre[kPrefetchVec];
    float pre_eta = 0.f;
    auto fetch = [&](int n0) {   // this thread's vectors (and eta) of mini-batch n0 into registers
        if (tid < mb) pre_eta = eg[n0 + tid];
#pragma unroll
        for (int r = 0; r < kPrefetchVec; ++r) {
            const int v = tid + r * kThreads;
            if (v < 3 * nt4) {
                const int which = v / nt4, i = (v - which * nt4) * 4;
                const IO *src = which == 0 ? Kg : which == 1 ? Qg : Vg;
                pre[r] = V4::load(src, (size_t)n0 * d + i);
            }
        }
    };
    auto stage = [&](int n0) {   // K, Q, V, eta of mini-batch n0 into shared memory (fp32)
        if (prefetch) {
#pragma unroll
            for (int r = 0; r < kPrefetchVec; ++r) {
                const int v = tid + r * kThreads;
                if (v < 3 * nt4) {
                    const int which = v / nt4, i = (v - which * nt4) * 4;
                    float *dst = which == 0 ? Kt : which == 1 ? Qt : Vt;
                    *reinterpret_cast<float4 *>(dst + i) = V4::to_f32(pre[r]);
                }
            }
            if (tid < mb) et[tid] = pre_eta;
        } else {
            for (int v = tid; v < 3 * nt4; v += kThreads) {
                const int which = v / nt4, i = (v - which * nt4) * 4;
                const IO *src = which == 0 ? Kg : which == 1 ? Qg : Vg;
                float *dst = which == 0 ? Kt : which == 1 ? Qt : Vt;
                *reinterpret_cast<float4 *>(dst + i) = V4::to_f32(V4::load(src, (size_t)n0 * d + i));
            }
            for (int s = tid; s < mb; s += kThreads) et[s] = eg[n0 + s];
        }
    };

    if (prefetch) fetch(0);
    for (int n0 = 0; n0 < L; n0 += mb) {
        __syncthreads();   // the previous mini-batch is done with the tiles
        stage(n0);
        __syncthreads();
        if (prefetch && n0 + mb < L) fetch(n0 + mb);
        // key- and query-side products at the mini-batch's starting weights: thread tile =
        // 4 features of one token, both sides; with weight decay the query row t sees
        // (1 - lambda sum_{s<=t} eta_s) W_start
        for (int tile = tid; tile < nt4; tile += kThreads) {
            const int t = tile / d4, j = (tile - t * d4) * 4;
            float4 ak = f4(c + j), aq = make_float4(0.f, 0.f, 0.f, 0.f);
            const float *kr = Kt + t * d, *qr = Qt + t * d;
#pragma unroll(DC ? DC / 4 : 1)
            for (int u = 0; u < d; u += 4) {
                const float4 k4 = f4(kr + u), q4 = f4(qr + u);
                const float4 w0 = f4(W + u * d + j), w1 = f4(W + (u + 1) * d + j);
                const float4 w2 = f4(W + (u + 2) * d + j), w3 = f4(W + (u + 3) * d + j);
                fma4(ak, k4.x, w0); fma4(ak, k4.y, w1); fma4(ak, k4.z, w2); fma4(ak, k4.w, w3);
                fma4(aq, q4.x, w0); fma4(aq, q4.y, w1); fma4(aq, q4.z, w2); fma4(aq, q4.w, w3);
            }
            *reinterpret_cast<float4 *>(G + t * d + j) = ak;
            const float f = 1.f - p.wd * eta_prefix(et, t);
            const float4 cj = f4(c + j);
            *reinterpret_cast<float4 *>(Zb + t * d + j) =
                make_float4(fmaf(f, aq.x, cj.x), fmaf(f, aq.y, cj.y), fmaf(f, aq.z, cj.z), fmaf(f, aq.w, cj.w));
        }
        // A[t, s] = eta_s (q_t . k_s + 1), s <= t.  Neighbouring threads take neighbouring s,
        // whose K rows are d floats apart: each starts its dot product 4 s columns further on
        // (wrapping), so their 16-byte loads fall in different shared-memory banks.
        for (int i = tid; i < mb * mb; i += kThreads) {
            const int t = i / mb, s = i - t * mb;
            float a = 0.f;
            if (s <= t) {
                const float *qr = Qt + t * d, *kr = Kt + s * d;
                float a0 = 0.f, a1 = 0.f;
                int u = (4 * s) % d;
#pragma unroll(DC ? DC / 4 : 1)
                for (int c = 0; c < d; c += 4) {
                    const float4 q4 = f4(qr + u), k4 = f4(kr + u);
                    a0 = fmaf(q4.x, k4.x, a0);
                    a1 = fmaf(q4.y, k4.y, a1);
                    a0 = fmaf(q4.z, k4.z, a0);
                    a1 = fmaf(q4.w, k4.w, a1);
                    u += 4;
                    if (u >= d) u -= d;
                }
                a = (a0 + a1 + 1.f) * et[s];
            }
            A[i] = a;
        }
        __syncthreads();
        if (LN) {
            for (int s = warp; s < mb; s += kWarps) {
                if (p.ip)
                    ln_ip_bwd_row(G + s * d, Vt + s * d, gam, d, p.eps);
                else
                    ln_l2_bwd_row(G + s * d, Vt + s * d, Kt + s * d, gam, bet, d, p.eps);
            }
        } else {
            for (int i = tid; i < nt; i += kThreads) G[i] = p.ip ? -Vt[i] : G[i] - Vt[i];
        }
        __syncthreads();
        // dual-form outputs: Zb[t] -= sum_{s <= t} A[t, s] G[s]   (4 features of one token)
        for (int tile = tid; tile < nt4; tile += kThreads) {
            const int t = tile / d4, j = (tile - t * d4) * 4;
            float4 z = f4(Zb + t * d + j);
            for (int s = 0; s <= t; ++s) fma4(z, -A[t * mb + s], f4(G + s * d + j));
            if (LN) {
                *reinterpret_cast<float4 *>(Zb + t * d + j) = z;
            } else {
                const size_t o = (size_t)(n0 + t) * d + j;
                store_io(Zg, o, z.x);
                store_io(Zg, o + 1, z.y);
                store_io(Zg, o + 2, z.z);
                store_io(Zg, o + 3, z.w);
            }
        }
        // carry: W <- (1 - lambda sum eta) W - K^T diag(eta) G (4 x 4 blocks of W),
        // c -= eta^T G
        const float decay = 1.f - p.wd * eta_prefix(et, mb - 1);
        for (int tile = tid; tile < d4 * d4; tile += kThreads) {
            const int u = (tile / d4) * 4, j = (tile - (tile / d4) * d4) * 4;
            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
            for (int s = 0; s < mb; ++s) {
                const float e = et[s];
                const float4 k4 = f4(Kt + s * d + u), g4 = f4(G + s * d + j);
                fma4(a0, e * k4.x, g4);
                fma4(a1, e * k4.y, g4);
                fma4(a2, e * k4.z, g4);
                fma4(a3, e * k4.w, g4);
            }
            const float4 acc[4] = {a0, a1, a2, a3};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float4 x = *reinterpret_cast<float4 *>(W + (u + r) * d + j);
                x.x = fmaf(decay, x.x, -acc[r].x);
                x.y = fmaf(decay, x.y, -acc[r].y);
                x.z = fmaf(decay, x.z, -acc[r].z);
                x.w = fmaf(decay, x.w, -acc[r].w);
                *reinterpret_cast<float4 *>(W + (u + r) * d + j) = x;
            }
        }
        for (int j = tid; j < d; j += kThreads) {
            float acc = 0.f;
            for (int s = 0; s < mb; ++s) acc = fmaf(et[s], G[s * d + j], acc);
            c[j] -= acc;
        }
        if (LN) {
            __syncthreads();
            for (int t = warp; t < mb; t += kWarps)
                ln_out_row(Zb + t * d, Qt + t * d, gam, bet, d, p.eps, Zg + (size_t)(n0 + t) * d);
        }
    }
    __syncthreads();
    for (int i = tid; i < d * d; i += kThreads) p.Wf[(size_t)bh * d * d + i] = W[i];
    for (int j = tid; j < d; j += kThreads) p.bf[(size_t)bh * d + j] = c[j] + pivot;
}

// ---------------------------------------------------------------------------
// TTT-MLP
// ---------------------------------------------------------------------------
struct MlpParams {
    int H, L, d, dh, mb, ln, init_per_batch;
    float eps;
    int ip;                  // inner-product loss
    float wd;                // weight decay lambda
    const void *Q, *K, *V;
    const float *eta, *W1, *b1, *W2, *b2, *gamma, *beta;
    void *Z;
    float *W1f, *b1f, *W2f, *b2f;
    int hoff = 0;            // head index of row 0 of this call
};

template <typename IO, bool LN>
__global__ void __launch_bounds__(kThreads) mlp_generic_kernel(MlpParams p)
{
    extern __shared__ float sm[];
    const int d = p.d, dh = p.dh, mb = p.mb, L = p.L;
    const int bh = blockIdx.x, h = (p.hoff + bh) % p.H;
    const int tid = threadIdx.x, warp = tid >> 5;
    float *W1 = sm;               // d*dh
    float *W2 = W1 + d * dh;      // dh*d
    float *b1 = W2 + dh * d;      // dh
    float *b2 = b1 + dh;          // d
    float *Kt = b2 + d;           // mb*d
    float *Qt = Kt + mb * d;
    float *Vt = Qt + mb * d;
    float *Z1 = Vt + mb * d;      // mb*dh : Z1, then G1
    float *X2 = Z1 + mb * dh;     // mb*dh
    float *Zb1 = X2 + mb * dh;    // mb*dh : Zb1, then Xb2
    float *Z2 = Zb1 + mb * dh;    // mb*d  : Z2, then G2
    float *Zb2 = Z2 + mb * d;     // mb*d
    float *A = Zb2 + mb * d;      // mb*mb
    float *et = A + mb * mb;      // mb
    float *gam = et + mb;         // d
    float *bet = gam + d;         // d

    const size_t init = p.init_per_batch ? (size_t)bh : (size_t)h;
    for (int i = tid; i < d * dh; i += kThreads) {
        W1[i] = p.W1[init * d * dh + i];
        W2[i] = p.W2[init * d * dh + i];
    }
    for (int m = tid; m < dh; m += kThreads) b1[m] = p.b1[init * dh + m];
    for (int j = tid; j < d; j += kThreads) {
        b2[j] = p.b2[init * d + j];
        if (LN) {
            gam[j] = p.gamma[(size_t)h * d + j];
            bet[j] = p.beta[(size_t)h * d + j];
        }
    }
    // LayerNorm pivot (as in the linear kernel): the scan runs on b2 - mean(b2)
    const float pivot = LN ? shift_by_mean(b2, d) : 0.f;
    const IO *Qg = static_cast<const IO *>(p.Q) + (size_t)bh * L * d;
    const IO *Kg = static_cast<const IO *>(p.K) + (size_t)bh * L * d;
    const IO *Vg = static_cast<const IO *>(p.V) + (size_t)bh * L * d;
    IO *Zg = static_cast<IO *>(p.Z) + (size_t)bh * L * d;
    const float *eg = p.eta + (size_t)bh * L;
    const int nt = mb * d, nh = mb * dh;

    for (int n0 = 0; n0 < L; n0 += mb) {
        __syncthreads();
        for (int i = tid; i < nt; i += kThreads) {
            size_t gi = (size_t)n0 * d + i;
            Kt[i] = load_io(Kg, gi);
            Qt[i] = load_io(Qg, gi);
            Vt[i] = load_io(Vg, gi);
        }
        for (int s = tid; s < mb; s += kThreads) et[s] = eg[n0 + s];
        __syncthreads();
        // first layer at the starting weights, key and query side
        for (int i = tid; i < nh; i += kThreads) {
            const int s = i / dh, m = i - s * dh;
            float ak = b1[m], aq = 0.f;
            for (int u = 0; u < d; ++u) {
                const float w = W1[u * dh + m];
                ak = fmaf(Kt[s * d + u], w, ak);
                aq = fmaf(Qt[s * d + u], w, aq);
            }
            Z1[i] = ak;
            X2[i] = gelu_tanh(ak);
            Zb1[i] = fmaf(1.f - p.wd * eta_prefix(et, s), aq, b1[m]);
        }
        for (int i = tid; i < mb * mb; i += kThreads) {
            const int t = i / mb, s = i - t * mb;
            float a = 0.f;
            if (s <= t) {
                for (int u = 0; u < d; ++u) a = fmaf(Qt[t * d + u], Kt[s * d + u], a);
                a = (a + 1.f) * et[s];
            }
            A[i] = a;
        }
        __syncthreads();
        // second layer, key side
        for (int i = tid; i < nt; i += kThreads) {
            const int s = i / d, j = i - s * d;
            float a = b2[j];
            for (int m = 0; m < dh; ++m) a = fmaf(X2[s * dh + m], W2[m * d + j], a);
            Z2[i] = a;
        }
        __syncthreads();
        if (LN) {
            for (int s = warp; s < mb; s += kWarps) {
                if (p.ip)
                    ln_ip_bwd_row(Z2 + s * d, Vt + s * d, gam, d, p.eps);
                else
                    ln_l2_bwd_row(Z2 + s * d, Vt + s * d, Kt + s * d, gam, bet, d, p.eps);
            }
        } else {
            for (int i = tid; i < nt; i += kThreads) Z2[i] = p.ip ? -Vt[i] : Z2[i] - Vt[i];
        }
        __syncthreads();
        // G1 = (G2 W2^T) * GELU'(Z1), in place over Z1; query side of layer 1
        for (int i = tid; i < nh; i += kThreads) {
            const int s = i / dh, m = i - s * dh;
            float a = 0.f;
            for (int j = 0; j < d; ++j) a = fmaf(Z2[s * d + j], W2[m * d + j], a);
            Z1[i] = a * gelu_tanh_prime(Z1[i]);
        }
        __syncthreads();
        for (int i = tid; i < nh; i += kThreads) {
            const int t = i / dh, m = i - t * dh;
            float z = Zb1[i];
            for (int s = 0; s <= t; ++s) z = fmaf(-A[t * mb + s], Z1[s * dh + m], z);
            Zb1[i] = gelu_tanh(z);  // Xb2
        }
        __syncthreads();
        for (int i = tid; i < mb * mb; i += kThreads) {
            const int t = i / mb, s = i - t * mb;
            float a = 0.f;
            if (s <= t) {
                for (int m = 0; m < dh; ++m) a = fmaf(Zb1[t * dh + m], X2[s * dh + m], a);
                a = (a + 1.f) * et[s];
            }
            A[i] = a;
        }
        __syncthreads();
        for (int i = tid; i < nt; i += kThreads) {
            const int t = i / d, j = i - t * d;
            float z = 0.f;
            for (int m = 0; m < dh; ++m) z = fmaf(Zb1[t * dh + m], W2[m * d + j], z);
            z = fmaf(1.f - p.wd * eta_prefix(et, t), z, b2[j]);
            for (int s = 0; s <= t; ++s) z = fmaf(-A[t * mb + s], Z2[s * d + j], z);
            if (LN)
                Zb2[i] = z;
            else
                store_io(Zg, (size_t)(n0 + t) * d + j, z);
        }
        __syncthreads();
        // carry (weight decay scales W1 and W2 by 1 - lambda sum eta)
        const float decay = 1.f - p.wd * eta_prefix(et, mb - 1);
        for (int i = tid; i < d * dh; i += kThreads) {
            const int u = i / dh, m = i - u * dh;
            float acc = 0.f;
            for (int s = 0; s < mb; ++s) acc = fmaf(et[s] * Kt[s * d + u], Z1[s * dh + m], acc);
            W1[i] = fmaf(decay, W1[i], -acc);
        }
        for (int i = tid; i < dh * d; i += kThreads) {
            const int m = i / d, j = i - m * d;
            float acc = 0.f;
            for (int s = 0; s < mb; ++s) acc = fmaf(et[s] * X2[s * dh + m], Z2[s * d + j], acc);
            W2[i] = fmaf(decay, W2[i], -acc);
        }
        for (int m = tid; m < dh; m += kThreads) {
            float acc = 0.f;
            for (int s = 0; s < mb; ++s) acc = fmaf(et[s], Z1[s * dh + m], acc);
            b1[m] -= acc;
        }
        for (int j = tid; j < d; j += kThreads) {
            float acc = 0.f;
            for (int s = 0; s < mb; ++s) acc = fmaf(et[s], Z2[s * d + j], acc);
            b2[j] -= acc;
        }
        if (LN) {
            for (int t = warp; t < mb; t += kWarps)
                ln_out_row(Zb2 + t * d, Qt + t * d, gam, bet, d, p.eps, Zg + (size_t)(n0 + t) * d);
        }
    }
    __syncthreads();
    for (int i = tid; i < d * dh; i += kThreads) {
        p.W1f[(size_t)bh * d * dh + i] = W1[i];
        p.W2f[(size_t)bh * d * dh + i] = W2[i];
    }
    for (int m = tid; m < dh; m += kThreads) p.b1f[(size_t)bh * dh + m] = b1[m];
    for (int j = tid; j < d; j += kThreads) p.b2f[(size_t)bh * d + j] = b2[j] + pivot;
}

constexpr size_t kMaxSmem = 227 * 1024;

template <typename K>
cudaError_t launch(K kernel, int grid, size_t smem, cudaStream_t stream, const void *params)
{
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {const_cast<void *>(params)};
    return cudaLaunchKernel((const void *)kernel, dim3(grid), dim3(kThreads), args, smem, stream);
}

}  // namespace

size_t linear_generic_smem_bytes(const ttt_desc &s)
{
    if (s.d > 128 || s.d % 4 != 0 || s.mini_batch > 64) return 0;
    size_t d = s.d, mb = s.mini_batch;
    size_t n = d * d + d + 5 * mb * d + mb * mb + mb + 2 * d;
    size_t bytes = n * sizeof(float);
    return bytes <= kMaxSmem ? bytes : 0;
}

cudaError_t launch_linear_generic(const LinearArgs &a)
{
    const ttt_desc &s = a.desc;
    LinearParams p{s.H, s.L, s.d, s.mini_batch, s.residual_ln, s.init_per_batch, s.ln_eps,
                   s.loss == TTT_LOSS_INNER_PRODUCT, s.weight_decay,
                   a.Q, a.K, a.V, a.eta, a.W0, a.b0, a.gamma, a.beta, a.Z, a.W_final, a.b_final};
    p.hoff = head_offset(s);
    const size_t smem = linear_generic_smem_bytes(s);
    const int grid = call_rows(s);
    const bool f32 = s.io_dtype == TTT_F32, ln = s.residual_ln != 0, d64 = s.d == 64;
    auto pick = [&](auto k64, auto kany) { return d64 ? (const void *)k64 : (const void *)kany; };
    const void *k = f32 ? (ln ? pick(linear_generic_kernel<float, true, 64>, linear_generic_kernel<float, true, 0>)
                              : pick(linear_generic_kernel<float, false, 64>, linear_generic_kernel<float, false, 0>))
                        : (ln ? pick(linear_generic_kernel<__nv_bfloat16, true, 64>,
                                     linear_generic_kernel<__nv_bfloat16, true, 0>)
                              : pick(linear_generic_kernel<__nv_bfloat16, false, 64>,
                                     linear_generic_kernel<__nv_bfloat16, false, 0>));
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {&p};
    return cudaLaunchKernel(k, dim3(grid), dim3(kLinThreads), args, smem, a.stream);
}

size_t mlp_generic_smem_bytes(const ttt_desc &s)
{
    if (s.d > 128 || s.d_hidden > 512 || s.mini_batch > 64) return 0;
    size_t d = s.d, dh = s.d_hidden, mb = s.mini_batch;
    size_t n = 2 * d * dh + dh + d + 3 * mb * d + 3 * mb * dh + 2 * mb * d + mb * mb + mb + 2 * d;
    size_t bytes = n * sizeof(float);
    return bytes <= kMaxSmem ? bytes : 0;
}

cudaError_t launch_mlp_generic(const MlpArgs &a)
{
    const ttt_desc &s = a.desc;
    MlpParams p{s.H, s.L, s.d, s.d_hidden, s.mini_batch, s.residual_ln, s.init_per_batch, s.ln_eps,
                s.loss == TTT_LOSS_INNER_PRODUCT, s.weight_decay,
                a.Q, a.K, a.V, a.eta, a.W1_0, a.b1_0, a.W2_0, a.b2_0, a.gamma, a.beta, a.Z,
                a.W1_f, a.b1_f, a.W2_f, a.b2_f};
    p.hoff = head_offset(s);
    const size_t smem = mlp_generic_smem_bytes(s);
    const int grid = call_rows(s);
    if (s.io_dtype == TTT_F32)
        return s.residual_ln ? launch(mlp_generic_kernel<float, true>, grid, smem, a.stream, &p)
                             : launch(mlp_generic_kernel<float, false>, grid, smem, a.stream, &p);
    return s.residual_ln ? launch(mlp_generic_kernel<__nv_bfloat16, true>, grid, smem, a.stream, &p)
                         : launch(mlp_generic_kernel<__nv_bfloat16, false>, grid, smem, a.stream, &p);
}

}  // namespace ttt
