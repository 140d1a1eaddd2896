// ttt_backward.cu -- backward pass of the TTT-Linear inner loop (with or without the residual
// LayerNorm, either loss, optional weight decay).
//
// Training through the inner loop (the meta-learning gradient of the damodev.csdn.net TTT
// article, section 6.1) needs the vector-Jacobian product of the mini-batch scan of
// sections 4.1-4.2: given dZ and the gradients dW_final, db_final of the final state,
// the gradients of Q, K, V, eta, W0, b0.  Per mini-batch n, with E = diag(eta_n), the
// causal mask M (s <= t) and the forward
//   P = K W + 1 c,  G = P - V  (inner-product loss: G = -V),
//   A = M . (Q K^T + 1) E,  Z = Q W + 1 c - A G,
//   W' = W - K^T E G,  c' = c - G^T eta,
// the reverse step from the gradients dW', dc' of the state after the mini-batch is
//   dG  = -A^T dZ - E K dW' - eta dc'^T,          D = M . (dZ G^T)
//   dQ  = dZ W^T - D E K
//   dK  = dG W^T - E G dW'^T - E D^T Q             (the dG W^T term: squared-error loss)
//   dV  = -dG
//   deta_s = -(K dW')_s . g_s - g_s . dc' - sum_t D[t, s] (q_t . k_s + 1)
//   dW  = dW' + Q^T dZ + K^T dG,   dc = dc' + 1^T dZ + 1^T dG   (K^T dG, 1^T dG: squared error)
// and dW, dc are the gradients of the state before the mini-batch.  With the residual
// LayerNorm dZ above is the output LayerNorm's backward of dZ (dQ also gets dZ itself), and G's
// dependence on P and on v (and k) is taken through the per-token Hessian-vector product of
// the LN-L2 loss.  With weight decay lambda (W' = (1 - lambda S) W - ..., query row t reading
// (1 - lambda cum_t) W, ai-feeds Modular TTT page): dW' is scaled by 1 - lambda S, Q^T dZ and
// dZ W^T by 1 - lambda cum_t per token, and
//   deta_s gains -lambda <W, dW'> - lambda sum_{t >= s} <dZ_t, q_t W>.  The scan reads the
// states in reverse, so the kernel first re-runs the forward and checkpoints the state
// every `ck` mini-batches in the workspace; the reverse pass restores a chunk's states
// from its checkpoint in shared memory and walks its mini-batches backwards.
//
// B300 design: one CTA per (batch, head), 256 threads, fp32 FFMA on shared-memory tiles
// (register-tiled loops with 16-byte loads).  For d = 64, b = 16 the tiles of the next
// forward or reverse step (its K, V or K, Q, V, dZ rows and eta) are copied global -> shared
// with cp.async while the current step computes: the order of the steps is fixed (pass 1,
// then per chunk the re-runs and the reverse steps), so the next one is always known.  The gradients of a head-shared initial state
// are summed over the batch by a second kernel, in a fixed order (deterministic).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float load_io(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_io(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void store_io(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_io(__nv_bfloat16 *p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

__device__ __forceinline__ float4 f4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void fma4(float4 &a, float s, float4 b)
{
    a.x = fmaf(s, b.x, a.x);
    a.y = fmaf(s, b.y, a.y);
    a.z = fmaf(s, b.z, a.z);
    a.w = fmaf(s, b.w, a.w);
}
__device__ __forceinline__ float dot4(float4 a, float4 b) { return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w))); }

// out[r][j..j+3] = init[j..j+3] + sum_u X[r][u] Y[u][j..j+3]   (X: m x k, Y: k x n, row-major;
// n, k multiples of 4; init may be null)
__device__ __forceinline__ void mm_xy(float *out, const float *X, const float *Y, const float *init, int m, int k,
                                      int n)
{
    const int n4 = n >> 2;
    if ((m & 1) == 0 && (k & 7) == 0 && n4 == 16 && (m >> 1) * n4 * 2 == kThreads) {
        // A 2 x 4 block (rows r, r + 1; columns j..j+3) per pair of lanes l, l + 16, each lane
        // summing one half of k: 6 shared loads per 32 FMAs instead of 5 per 16.  The 16 lanes
        // of a half read one 256-byte row of Y, so no two lanes of a quarter-warp share a bank;
        // one shuffle adds the halves, and each lane of the pair stores one row.
        const int lane = threadIdx.x & 31, half = lane >> 4;
        const int r = (threadIdx.x >> 5) * 2, j = (lane & 15) * 4;
        const int kh = k >> 1, u0 = half * kh;
        const float *x0 = X + r * k, *x1 = x0 + k;
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
        for (int u = u0; u < u0 + kh; u += 4) {
            const float4 xa = f4(x0 + u), xb = f4(x1 + u);
            const float4 w0 = f4(Y + u * n + j), w1 = f4(Y + (u + 1) * n + j);
            const float4 w2 = f4(Y + (u + 2) * n + j), w3 = f4(Y + (u + 3) * n + j);
            fma4(a0, xa.x, w0); fma4(a0, xa.y, w1); fma4(a0, xa.z, w2); fma4(a0, xa.w, w3);
            fma4(a1, xb.x, w0); fma4(a1, xb.y, w1); fma4(a1, xb.z, w2); fma4(a1, xb.w, w3);
        }
        a0.x += __shfl_xor_sync(0xffffffffu, a0.x, 16);
        a0.y += __shfl_xor_sync(0xffffffffu, a0.y, 16);
        a0.z += __shfl_xor_sync(0xffffffffu, a0.z, 16);
        a0.w += __shfl_xor_sync(0xffffffffu, a0.w, 16);
        a1.x += __shfl_xor_sync(0xffffffffu, a1.x, 16);
        a1.y += __shfl_xor_sync(0xffffffffu, a1.y, 16);
        a1.z += __shfl_xor_sync(0xffffffffu, a1.z, 16);
        a1.w += __shfl_xor_sync(0xffffffffu, a1.w, 16);
        float4 a = half ? a1 : a0;
        if (init) {
            const float4 b = f4(init + j);
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        st4(out + (r + half) * n + j, a);
        return;
    }
    for (int tile = threadIdx.x; tile < m * n4; tile += kThreads) {
        const int r = tile / n4, j = (tile - r * n4) * 4;
        float4 a = init ? f4(init + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float *xr = X + r * k;
#pragma unroll
        for (int u = 0; u < k; u += 4) {
            const float4 x = f4(xr + u);
            fma4(a, x.x, f4(Y + u * n + j));
            fma4(a, x.y, f4(Y + (u + 1) * n + j));
            fma4(a, x.z, f4(Y + (u + 2) * n + j));
            fma4(a, x.w, f4(Y + (u + 3) * n + j));
        }
        st4(out + r * n + j, a);
    }
}

// The same with two left factors sharing Y: outA = XA Y + initA, outB = XB Y (one read of
// each Y row serves both products)
__device__ __forceinline__ void mm_xy2(float *outA, float *outB, const float *XA, const float *XB, const float *Y,
                                      const float *initA, int m, int k, int n)
{
    const int n4 = n >> 2;
    if ((m & 1) == 0 && (k & 7) == 0 && n4 == 16 && (m >> 1) * n4 * 2 == kThreads) {
        // rows r, r + 1 of both products per pair of lanes l, l + 16 splitting k (as in mm_xy):
        // 8 shared loads per 64 FMAs
        const int lane = threadIdx.x & 31, half = lane >> 4;
        const int r = (threadIdx.x >> 5) * 2, j = (lane & 15) * 4;
        const int kh = k >> 1, u0 = half * kh;
        const float *xa = XA + r * k, *xb = XB + r * k;
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
#pragma unroll
        for (int u = u0; u < u0 + kh; u += 4) {
            const float4 p0 = f4(xa + u), p1 = f4(xa + k + u), q0 = f4(xb + u), q1 = f4(xb + k + u);
            const float4 w0 = f4(Y + u * n + j), w1 = f4(Y + (u + 1) * n + j);
            const float4 w2 = f4(Y + (u + 2) * n + j), w3 = f4(Y + (u + 3) * n + j);
            fma4(a0, p0.x, w0); fma4(a0, p0.y, w1); fma4(a0, p0.z, w2); fma4(a0, p0.w, w3);
            fma4(a1, p1.x, w0); fma4(a1, p1.y, w1); fma4(a1, p1.z, w2); fma4(a1, p1.w, w3);
            fma4(b0, q0.x, w0); fma4(b0, q0.y, w1); fma4(b0, q0.z, w2); fma4(b0, q0.w, w3);
            fma4(b1, q1.x, w0); fma4(b1, q1.y, w1); fma4(b1, q1.z, w2); fma4(b1, q1.w, w3);
        }
        // each lane keeps (and stores) its own row: row r on the low half, r + 1 on the high one
        float4 a = half ? a1 : a0, b = half ? b1 : b0;
        const float4 ao = half ? a0 : a1, bo = half ? b0 : b1;   // the partner's row, sent over
        a.x += __shfl_xor_sync(0xffffffffu, ao.x, 16);
        a.y += __shfl_xor_sync(0xffffffffu, ao.y, 16);
        a.z += __shfl_xor_sync(0xffffffffu, ao.z, 16);
        a.w += __shfl_xor_sync(0xffffffffu, ao.w, 16);
        b.x += __shfl_xor_sync(0xffffffffu, bo.x, 16);
        b.y += __shfl_xor_sync(0xffffffffu, bo.y, 16);
        b.z += __shfl_xor_sync(0xffffffffu, bo.z, 16);
        b.w += __shfl_xor_sync(0xffffffffu, bo.w, 16);
        if (initA) {
            const float4 c = f4(initA + j);
            a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
        }
        st4(outA + (r + half) * n + j, a);
        st4(outB + (r + half) * n + j, b);
        return;
    }
    for (int tile = threadIdx.x; tile < m * n4; tile += kThreads) {
        const int r = tile / n4, j = (tile - r * n4) * 4;
        float4 a = initA ? f4(initA + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
        const float *xa = XA + r * k, *xb = XB + r * k;
#pragma unroll
        for (int u = 0; u < k; u += 4) {
            const float4 x = f4(xa + u), y = f4(xb + u);
            const float4 w0 = f4(Y + u * n + j), w1 = f4(Y + (u + 1) * n + j);
            const float4 w2 = f4(Y + (u + 2) * n + j), w3 = f4(Y + (u + 3) * n + j);
            fma4(a, x.x, w0); fma4(a, x.y, w1); fma4(a, x.z, w2); fma4(a, x.w, w3);
            fma4(b, y.x, w0); fma4(b, y.y, w1); fma4(b, y.z, w2); fma4(b, y.w, w3);
        }
        st4(outA + r * n + j, a);
        st4(outB + r * n + j, b);
    }
}

// Dot product of two k-long shared-memory rows, starting at column `start` (a multiple of 4)
// and wrapping: threads whose rows are k floats apart start 4 floats apart, so their 16-byte
// loads fall in different banks.
__device__ __forceinline__ float rot_dot(const float *x, const float *y, int k, int start)
{
    float a0 = 0.f, a1 = 0.f;
    int u = start;
#pragma unroll
    for (int c = 0; c < k; c += 8) {
        a0 += dot4(f4(x + u), f4(y + u));
        u += 4;
        if (u >= k) u -= k;
        if (c + 4 < k) {
            a1 += dot4(f4(x + u), f4(y + u));
            u += 4;
            if (u >= k) u -= k;
        }
    }
    return a0 + a1;
}
__device__ __forceinline__ int rot_start(int row, int k) { return (4 * row) % k; }

// out[r][i] = sum_j X[r][j] Y[i][j]   (X Y^T; X: m x k, Y: n x k; k a multiple of 4).
// With m and n even each thread takes a 2 x 2 block (rows r, r + 1 of X against rows i, i + 1
// of Y): four independent sums and two loads per four products; neighbouring threads take
// neighbouring row pairs of Y, each starting 4 columns further on (wrapping), so their
// 16-byte loads fall in different banks.
__device__ __forceinline__ void mm_xyt(float *out, const float *X, const float *Y, int m, int k, int n)
{
    if ((m & 1) == 0 && (k & 7) == 0 && n == 64 && (m >> 1) * (n >> 2) * 2 == kThreads) {
        // A 2 x 4 block (rows r, r + 1 of X against rows i..i+3 of Y) per pair of lanes l, l + 16,
        // each lane summing one half of k: 6 loads per 32 FMAs instead of 4 per 16.  Each lane
        // starts its half at column 4 (l mod 8), wrapping, so the eight lanes of a quarter-warp
        // read eight different banks; one shuffle adds the halves, each lane stores one row.
        const int lane = threadIdx.x & 31, half = lane >> 4, q = lane & 15;
        const int r = (threadIdx.x >> 5) * 2, i = q * 4;
        const int kh = k >> 1;
        const float *x0 = X + r * k + half * kh, *x1 = x0 + k, *y0 = Y + i * k + half * kh;
        float a[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        int u = (4 * (q & 7)) % kh;
#pragma unroll
        for (int c = 0; c < kh; c += 4) {
            const float4 xa = f4(x0 + u), xb = f4(x1 + u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 y = f4(y0 + e * k + u);
                a[0][e] += dot4(xa, y);
                a[1][e] += dot4(xb, y);
            }
            u += 4;
            if (u >= kh) u -= kh;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) a[h][e] += __shfl_xor_sync(0xffffffffu, a[h][e], 16);
        st4(out + (r + half) * n + i, half ? make_float4(a[1][0], a[1][1], a[1][2], a[1][3])
                                           : make_float4(a[0][0], a[0][1], a[0][2], a[0][3]));
        return;
    }
    if ((m | n) & 1) {
        for (int idx = threadIdx.x; idx < m * n; idx += kThreads) {
            const int r = idx / n, i = idx - r * n;
            out[idx] = rot_dot(X + r * k, Y + i * k, k, rot_start(i, k));
        }
        return;
    }
    const int np = n >> 1;
    for (int idx = threadIdx.x; idx < (m >> 1) * np; idx += kThreads) {
        const int r = (idx / np) * 2, i = (idx - (idx / np) * np) * 2;
        const float *x0 = X + r * k, *x1 = x0 + k, *y0 = Y + i * k, *y1 = y0 + k;
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        int u = rot_start(i >> 1, k);
#pragma unroll
        for (int c = 0; c < k; c += 4) {
            const float4 xa = f4(x0 + u), xb = f4(x1 + u), ya = f4(y0 + u), yb = f4(y1 + u);
            a00 += dot4(xa, ya);
            a01 += dot4(xa, yb);
            a10 += dot4(xb, ya);
            a11 += dot4(xb, yb);
            u += 4;
            if (u >= k) u -= k;
        }
        out[r * n + i] = a00;
        out[r * n + i + 1] = a01;
        out[(r + 1) * n + i] = a10;
        out[(r + 1) * n + i + 1] = a11;
    }
}

// acc[u][j..j+3] = scale acc + sign sum_s w_s X[s][u] Y[s][j..j+3]   (X^T diag(w) Y, 4 x 4
// blocks; X: m x k, Y: m x n; w may be null (1))
__device__ __forceinline__ void mm_xty_acc(float *acc, const float *X, const float *Y, const float *w, float sign,
                                           int m, int k, int n, float scale = 1.f)
{
    const int n4 = n >> 2, k4 = k >> 2;
    for (int tile = threadIdx.x; tile < k4 * n4; tile += kThreads) {
        const int u = (tile / n4) * 4, j = (tile - (tile / n4) * n4) * 4;
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
        for (int s = 0; s < m; ++s) {
            const float e = w ? w[s] : 1.f;
            const float4 x = f4(X + s * k + u), y = f4(Y + s * n + j);
            fma4(a0, e * x.x, y);
            fma4(a1, e * x.y, y);
            fma4(a2, e * x.z, y);
            fma4(a3, e * x.w, y);
        }
        const float4 a[4] = {a0, a1, a2, a3};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float4 o = f4(acc + (u + r) * n + j);
            o.x = fmaf(sign, a[r].x, scale * o.x);
            o.y = fmaf(sign, a[r].y, scale * o.y);
            o.z = fmaf(sign, a[r].z, scale * o.z);
            o.w = fmaf(sign, a[r].w, scale * o.w);
            st4(acc + (u + r) * n + j, o);
        }
    }
}

// floats of the block A, D, eta, f_t, reduction (rounded up to 4: the tiles after it are read
// as float4)
__host__ __device__ constexpr int small_floats(int mb) { return (2 * mb * mb + 2 * mb + kThreads / 32 + 3) & ~3; }

struct BwdParams {
    int H, L, d, mb, ck;      // ck: mini-batches per checkpoint
    int init_per_batch, ip;
    float eps, wd;            // wd: weight decay lambda
    const void *Q, *K, *V, *dZ;
    const float *eta, *W0, *b0, *gamma, *beta, *dWf, *dbf;
    void *dQ, *dK, *dV;
    float *deta, *dW0, *db0;  // dW0/db0: per (batch, head) (the partials when the state is head-shared)
    float *dgb;               // LN: per-row partials [rows][2 d] of dgamma, dbeta
    float *ckpt;              // [rows][nck][d d + d]
    int hoff;
    int pf_off;               // float offset of the prefetch buffer in shared memory (d = 64, b = 16)
};

template <typename IO>
__device__ __forceinline__ void load_tile(float *dst, const IO *src, int n)
{
    for (int i = threadIdx.x; i < n; i += kThreads) dst[i] = load_io(src, i);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kMaxPerLane = 4;   // d <= 128: features lane, lane + 32, ... of a row

// Per-token LayerNorm quantities of a row z (d features, lane owns j = lane + 32 i):
// xh = (z - mu) r with two-pass statistics.
struct LnRow {
    float xh[kMaxPerLane];
    float r;
};
__device__ __forceinline__ LnRow ln_row(const float *z, int d, float eps)
{
    const int lane = threadIdx.x & 31;
    LnRow o;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int j = lane + 32 * i;
        if (j < d) s += z[j];
    }
    const float mu = warp_sum(s) / d;
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int j = lane + 32 * i;
        o.xh[i] = j < d ? z[j] - mu : 0.f;
        v += o.xh[i] * o.xh[i];
    }
    o.r = rsqrtf(warp_sum(v) / d + eps);
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) o.xh[i] *= o.r;
    return o;
}

// Pi w = w - mean(w) - xh mean(xh w), in place over the lane's features
__device__ __forceinline__ void ln_pi(float *w, const float *xh, int d)
{
    const int lane = threadIdx.x & 31;
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
        if (lane + 32 * i < d) {
            s1 += w[i];
            s2 += xh[i] * w[i];
        }
    s1 = warp_sum(s1) / d;
    s2 = warp_sum(s2) / d;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) w[i] = w[i] - s1 - xh[i] * s2;
}

// The per-token gradient with the residual LayerNorm, for the row z = k W + c:
// G = r Pi gx with gx = a xh + c0, a = gamma^2, c0 = gamma (beta - (v - k)) (squared error) or
// a = 0, c0 = -gamma v (inner product).  Returns gx in gxo when asked.
__device__ __forceinline__ void ln_grad_row(float *G, const float *z, const float *k, const float *v,
                                            const float *gam, const float *bet, int d, float eps, bool ip,
                                            const LnRow &ln, float *gxo)
{
    const int lane = threadIdx.x & 31;
    float w[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int j = lane + 32 * i;
        float gx = 0.f;
        if (j < d) gx = ip ? -gam[j] * v[j] : gam[j] * (gam[j] * ln.xh[i] + bet[j] - (v[j] - k[j]));
        w[i] = gx;
        if (gxo) gxo[i] = gx;
    }
    ln_pi(w, ln.xh, d);
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int j = lane + 32 * i;
        if (j < d) G[j] = ln.r * w[i];
    }
    (void)z;
}

// DT, MT: the head dim and the mini-batch size as compile-time constants (0: taken from the
// parameters at run time).  With both fixed, tile decodes are shifts and the fixed-length
// loops (the d-long dot products, the b-long sums, the causal b x b loops as predicated full
// loops) unroll, so their shared-memory loads are issued back to back.
template <typename IO, bool LN, int DT, int MT>
__global__ void __launch_bounds__(kThreads, 1) linear_bwd_kernel(BwdParams p)
{
    extern __shared__ float4 sm4[];
    float *sm = reinterpret_cast<float *>(sm4);
    const int d = DT ? DT : p.d, mb = MT ? MT : p.mb, L = p.L, ck = p.ck, dd = d * d;
    const int sd = dd + d;                        // one state: W then c
    const int bh = blockIdx.x, h = (p.hoff + bh) % p.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kWarps = kThreads / 32;
    // rows per warp in the warp-per-row loops (a compile-time count for b = 16, so they unroll
    // and the rows' shuffle reductions interleave)
    const int kRowIters = MT ? (MT + kWarps - 1) / kWarps : (mb + kWarps - 1) / kWarps;
    const int nmb = L / mb, nck = (nmb + ck - 1) / ck;
    const int nt = mb * d;
    const float kf = p.ip ? 0.f : 1.f;

    float *S = sm;                  // ck states [ck][d d + d]
    float *dW = S + ck * sd;        // d d, then dc (d)
    float *dc = dW + dd;
    float *Kt = dc + d;             // mb d each
    float *Qt = Kt + nt;
    float *Vt = Qt + nt;            // V; with LN later dy (dV)
    float *dZt = Vt + nt;
    float *G = dZt + nt;
    float *dG = G + nt;
    float *T1 = dG + nt;            // dZbar W^T, later dP W^T
    float *T2 = T1 + nt;            // K dW', later dP
    float *T3 = T2 + nt;            // G dW'^T
    // the layout below is mirrored by smem_for(); change both together
    float *A = T3 + nt;             // mb mb: R = M . (Q K^T + 1) (A = R E)
    float *Dm = A + mb * mb;        // mb mb
    float *et = Dm + mb * mb;       // mb
    float *fq = et + mb;            // mb: 1 - lambda cum_t (1 without weight decay)
    float *wred = fq + mb;          // kWarps: a block reduction
    float *Pz = A + small_floats(mb);   // LN or weight decay: P = K W + c
    float *dZb = Pz + nt;           // LN or weight decay: Zbar, then dZbar
    float *gam = dZb + nt;          // d
    float *bet = gam + d;           // d
    const bool wdec = p.wd != 0.f;
    // Q W (no bias): with weight decay its own tile (read again for deta); with LN alone it is
    // read only before T1 is first written, so it shares T1
    float *Yq = wdec ? bet + d : T1;
    // kWarps x 2 d for the final dgamma / dbeta reduction: the state area once the scan is
    // done, or its own area when the states are smaller (d < 16)
    float *red = (2 * d * kWarps <= ck * sd) ? S : (wdec ? Yq + nt : bet + d);
    if (!LN) dZb = dZt;
    // d = 64, b = 16: the next step's rows arrive by cp.async in `pf` (raw I/O elements:
    // K, Q, V, dZ tiles, then eta), placed after the last region of the plan
    constexpr bool kAsync = DT != 0 && MT != 0;
    unsigned char *pf = reinterpret_cast<unsigned char *>(sm + p.pf_off);
    constexpr int kEs = sizeof(IO);

    const IO *Qg = static_cast<const IO *>(p.Q) + (size_t)bh * L * d;
    const IO *Kg = static_cast<const IO *>(p.K) + (size_t)bh * L * d;
    const IO *Vg = static_cast<const IO *>(p.V) + (size_t)bh * L * d;
    const IO *dZg = static_cast<const IO *>(p.dZ) + (size_t)bh * L * d;
    const float *eg = p.eta + (size_t)bh * L;
    float *ck_base = p.ckpt + (size_t)bh * nck * sd;
    if (LN)
        for (int j = tid; j < d; j += kThreads) {
            gam[j] = p.gamma[(size_t)h * d + j];
            bet[j] = p.beta[(size_t)h * d + j];
        }

    // G = dl/dz of the tile's rows, from P (in G on entry for the plain loss; in src for LN)
    auto gradient_rows = [&](float *Gout, const float *src) {
        if (LN) {
            #pragma unroll
            for (int s = warp, it_ = 0; it_ < kRowIters; s += kWarps, ++it_) {
                if (s >= mb) break;
                const LnRow ln = ln_row(src + s * d, d, p.eps);
                ln_grad_row(Gout + s * d, src + s * d, Kt + s * d, Vt + s * d, gam, bet, d, p.eps, p.ip != 0, ln,
                            nullptr);
            }
        } else {
            for (int i = tid; i < nt; i += kThreads) Gout[i] = fmaf(src[i], kf, -Vt[i]);
        }
    };

    // The steps in order, each with the rows it reads: forward step n (K, V, eta of
    // mini-batch n) in pass 1 (n = 0 .. nmb - 2) and as a re-run in pass 2, reverse step n
    // (K, Q, V, dZ, eta).  kind: 0 forward, 1 reverse, -1 none.
    struct Op {
        int kind, n;
    };
    auto first_of_chunk = [&](int ci) -> Op {
        const int m0 = ci * ck, mcount = min(ck, nmb - m0);
        return mcount > 1 ? Op{0, m0} : Op{1, m0};
    };
    // copy the rows of `op` into pf (each thread its 16-byte chunks; one commit group)
    auto prefetch = [&](Op op) {
        if (!kAsync || op.kind < 0) return;
        const size_t off = (size_t)op.n * mb * d;
        constexpr int tile_chunks = (MT * DT * kEs) / 16;
        const IO *src[4] = {Kg + off, Qg + off, Vg + off, dZg + off};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            if (op.kind == 0 && (w == 1 || w == 3)) continue;   // forward: K and V only
            for (int ch = tid; ch < tile_chunks; ch += kThreads)
                ptx::cp_async16(ptx::smem_addr(pf + (w * tile_chunks + ch) * 16),
                                reinterpret_cast<const unsigned char *>(src[w]) + ch * 16);
        }
        if (tid < MT / 4)
            ptx::cp_async16(ptx::smem_addr(pf + 4 * tile_chunks * 16 + tid * 16), eg + (size_t)op.n * mb + tid * 4);
        ptx::cp_async_commit();
    };
    // the rows of `op` into the fp32 tiles (from pf when prefetched), then prefetch `next`
    auto stage_op = [&](Op op, Op next) {
        const int n0 = op.n * mb;
        if (kAsync) {
            ptx::cp_async_wait_all();
            __syncthreads();   // every thread's copies have landed; the last step's readers are done
            const IO *pk = reinterpret_cast<const IO *>(pf);
            float *dst[4] = {Kt, Qt, Vt, dZt};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                if (op.kind == 0 && (w == 1 || w == 3)) continue;
                for (int i = tid; i < nt; i += kThreads) dst[w][i] = load_io(pk + w * nt, i);
            }
            for (int s = tid; s < mb; s += kThreads)
                et[s] = reinterpret_cast<const float *>(pf + 4 * nt * kEs)[s];
            __syncthreads();   // pf is free again
            prefetch(next);
        } else {
            __syncthreads();
            load_tile(Kt, Kg + (size_t)n0 * d, nt);
            if (op.kind == 1) load_tile(Qt, Qg + (size_t)n0 * d, nt);
            load_tile(Vt, Vg + (size_t)n0 * d, nt);
            if (op.kind == 1) load_tile(dZt, dZg + (size_t)n0 * d, nt);
            for (int s = tid; s < mb; s += kThreads) et[s] = eg[n0 + s];
            __syncthreads();
        }
    };

    // one forward mini-batch on the state X (in place): G, W -= K^T E G, c -= G^T eta
    auto forward_step = [&](float *X, int n, Op next) {
        stage_op(Op{0, n}, next);
        mm_xy(LN ? Pz : G, Kt, X, X + dd, mb, d, d);
        __syncthreads();
        gradient_rows(G, LN ? Pz : G);
        __syncthreads();
        float esum = 0.f;
        if (wdec)
            for (int s2 = 0; s2 < mb; ++s2) esum += et[s2];
        mm_xty_acc(X, Kt, G, et, -1.f, mb, d, d, 1.f - p.wd * esum);
        for (int j = tid; j < d; j += kThreads) {
            float a = 0.f;
#pragma unroll
            for (int s = 0; s < mb; ++s) a = fmaf(et[s], G[s * d + j], a);
            X[dd + j] -= a;
        }
    };

    // ---- pass 1: forward, checkpoint the state at the start of every ck mini-batches
    const size_t init = p.init_per_batch ? (size_t)bh : (size_t)h;
    for (int i = tid; i < dd; i += kThreads) S[i] = p.W0[init * dd + i];
    for (int j = tid; j < d; j += kThreads) S[dd + j] = p.b0[init * d + j];
    prefetch(nmb >= 2 ? Op{0, 0} : first_of_chunk(nck - 1));
    for (int n = 0; n < nmb; ++n) {
        if (n % ck == 0) {
            __syncthreads();
            float *dst = ck_base + (size_t)(n / ck) * sd;
            for (int i = tid; i < sd; i += kThreads) dst[i] = S[i];
        }
        if (n + 1 < nmb)   // the last state is never needed
            forward_step(S, n, n + 2 < nmb ? Op{0, n + 1} : first_of_chunk(nck - 1));
    }

    // ---- pass 2: reverse
    float dgam_acc[kMaxPerLane], dbet_acc[kMaxPerLane];   // this warp's tokens (LN)
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) dgam_acc[i] = dbet_acc[i] = 0.f;
    for (int i = tid; i < dd; i += kThreads) dW[i] = p.dWf ? p.dWf[(size_t)bh * dd + i] : 0.f;
    for (int j = tid; j < d; j += kThreads) dc[j] = p.dbf ? p.dbf[(size_t)bh * d + j] : 0.f;
    for (int ci = nck - 1; ci >= 0; --ci) {
        const int m0 = ci * ck, mcount = min(ck, nmb - m0);
        // restore the chunk's states S[0..mcount)
        __syncthreads();
        const float *src = ck_base + (size_t)ci * sd;
        for (int i = tid; i < sd; i += kThreads) S[i] = src[i];
        for (int m = 1; m < mcount; ++m) {
            __syncthreads();
            for (int i = tid; i < sd; i += kThreads) S[m * sd + i] = S[(m - 1) * sd + i];
            forward_step(S + m * sd, m0 + m - 1, m + 1 < mcount ? Op{0, m0 + m} : Op{1, m0 + mcount - 1});
        }
        for (int m = mcount - 1; m >= 0; --m) {
            const int n0 = (m0 + m) * mb;
            const float *W = S + m * sd, *c = W + dd;
            stage_op(Op{1, m0 + m}, m > 0 ? Op{1, m0 + m - 1} : (ci > 0 ? first_of_chunk(ci - 1) : Op{-1, 0}));
            // P (LN: kept in Pz), K dW', R = M . (Q K^T + 1); Q W (with LN or weight decay)
            if (LN || wdec)
                mm_xy2(LN ? Pz : G, Yq, Kt, Qt, W, c, mb, d, d);
            else
                mm_xy(G, Kt, W, c, mb, d, d);
            mm_xy(T2, Kt, dW, nullptr, mb, d, d);
            if (tid == 0) {   // f_t = 1 - lambda sum_{s <= t} eta_s
                float cum = 0.f;
                for (int t = 0; t < mb; ++t) {
                    cum += et[t];
                    fq[t] = 1.f - p.wd * cum;
                }
            }
            for (int i = tid; i < mb * mb; i += kThreads) {
                const int t = i / mb, s = i - t * mb;
                A[i] = s <= t ? rot_dot(Qt + t * d, Kt + s * d, d, rot_start(s, d)) + 1.f : 0.f;
            }
            __syncthreads();
            gradient_rows(G, LN ? Pz : G);
            __syncthreads();
            if (LN) {
                // Zbar = f_t Q W + c - A G, then dZbar = r Pi(gamma dZ) (output LayerNorm backward);
                // dgamma += dZ . xh_o, dbeta += dZ
                for (int tile = tid; tile < nt / 4; tile += kThreads) {
                    const int t = tile / (d / 4), j = (tile - t * (d / 4)) * 4;
                    const float4 y = f4(Yq + t * d + j), cj = f4(c + j);
                    const float f = fq[t];
                    float4 z = make_float4(fmaf(f, y.x, cj.x), fmaf(f, y.y, cj.y), fmaf(f, y.z, cj.z),
                                           fmaf(f, y.w, cj.w));
#pragma unroll
                    for (int s = 0; s < mb; ++s)
                        if (s <= t) fma4(z, -et[s] * A[t * mb + s], f4(G + s * d + j));
                    st4(dZb + t * d + j, z);
                }
                __syncthreads();
                #pragma unroll
                for (int t = warp, it_ = 0; it_ < kRowIters; t += kWarps, ++it_) {
                    if (t >= mb) break;
                    const LnRow lo = ln_row(dZb + t * d, d, p.eps);
                    float w[kMaxPerLane];
#pragma unroll
                    for (int i = 0; i < kMaxPerLane; ++i) {
                        const int j = lane + 32 * i;
                        const float dz = j < d ? dZt[t * d + j] : 0.f;
                        w[i] = j < d ? gam[j] * dz : 0.f;
                        dgam_acc[i] = fmaf(dz, lo.xh[i], dgam_acc[i]);
                        dbet_acc[i] += dz;
                    }
                    ln_pi(w, lo.xh, d);
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < kMaxPerLane; ++i) {
                        const int j = lane + 32 * i;
                        if (j < d) dZb[t * d + j] = lo.r * w[i];
                    }
                }
                __syncthreads();
            }
            // dZbar W^T, G dW'^T, D = M . (dZbar G^T), dG = -A^T dZbar - E K dW' - eta dc'^T
            mm_xyt(T1, dZb, W, mb, d, d);
            mm_xyt(T3, G, dW, mb, d, d);
            for (int i = tid; i < mb * mb; i += kThreads) {
                const int t = i / mb, s = i - t * mb;
                Dm[i] = s <= t ? rot_dot(dZb + t * d, G + s * d, d, rot_start(s, d)) : 0.f;
            }
            for (int tile = tid; tile < nt / 4; tile += kThreads) {
                const int s = tile / (d / 4), j = (tile - s * (d / 4)) * 4;
                float4 a = f4(T2 + s * d + j);
                const float4 dcj = f4(dc + j);
                a.x = -et[s] * (a.x + dcj.x);
                a.y = -et[s] * (a.y + dcj.y);
                a.z = -et[s] * (a.z + dcj.z);
                a.w = -et[s] * (a.w + dcj.w);
#pragma unroll
                for (int t = 0; t < mb; ++t)
                    if (t >= s) fma4(a, -et[s] * A[t * mb + s], f4(dZb + t * d + j));
                st4(dG + s * d + j, a);
            }
            __syncthreads();
            // dQ = dZ (residual LN) + dZbar W^T - D E K
            IO *dQg = static_cast<IO *>(p.dQ) + (size_t)bh * L * d + (size_t)n0 * d;
            IO *dKg = static_cast<IO *>(p.dK) + (size_t)bh * L * d + (size_t)n0 * d;
            IO *dVg = static_cast<IO *>(p.dV) + (size_t)bh * L * d + (size_t)n0 * d;
            for (int tile = tid; tile < nt / 4; tile += kThreads) {
                const int t = tile / (d / 4), j = (tile - t * (d / 4)) * 4;
                float4 a = f4(T1 + t * d + j);
                const float f = fq[t];
                a.x *= f; a.y *= f; a.z *= f; a.w *= f;
                if (LN) {
                    const float4 z = f4(dZt + t * d + j);
                    a.x += z.x; a.y += z.y; a.z += z.z; a.w += z.w;
                }
#pragma unroll
                for (int s = 0; s < mb; ++s)
                    if (s <= t) fma4(a, -Dm[t * mb + s] * et[s], f4(Kt + s * d + j));
                store_io(dQg, t * d + j, a.x);
                store_io(dQg, t * d + j + 1, a.y);
                store_io(dQg, t * d + j + 2, a.z);
                store_io(dQg, t * d + j + 3, a.w);
            }
            // deta_s = -(K dW')_s . g_s - g_s . dc' - sum_{t >= s} D[t, s] (q_t . k_s + 1)
            //          [- lambda <W, dW'> - lambda sum_{t >= s} <dZbar_t, q_t W>]
            float wdw = 0.f;
            if (wdec) {
                float part = 0.f;
                for (int i = tid; i < dd; i += kThreads) part = fmaf(W[i], dW[i], part);
                part = warp_sum(part);
                if (lane == 0) wred[warp] = part;
                #pragma unroll
                for (int t = warp, it_ = 0; it_ < kRowIters; t += kWarps, ++it_) {
                    if (t >= mb) break;   // <dZbar_t, q_t W>
                    float x = 0.f;
                    for (int u = lane; u < d; u += 32) x = fmaf(dZb[t * d + u], Yq[t * d + u], x);
                    x = warp_sum(x);
                    __syncwarp();
                    if (lane == 0) Yq[t * d] = x;   // row t of Q W is not read again: keep the dot there
                }
                __syncthreads();
                for (int w2 = 0; w2 < kWarps; ++w2) wdw += wred[w2];
            }
            // sixteen lanes per token s: lane i takes features i, i + 16, ... and targets
            // t = i, i + 16, ... (t >= s), then the sixteen partials are summed by shuffles
            for (int s0 = 0; s0 < mb; s0 += kThreads / 16) {
                const int s = s0 + tid / 16, i16 = tid & 15;
                float a = 0.f;
                if (s < mb) {
                    for (int u = i16; u < d; u += 16) a -= (T2[s * d + u] + dc[u]) * G[s * d + u];
                    for (int t = s + i16; t < mb; t += 16) {
                        a -= Dm[t * mb + s] * A[t * mb + s];
                        if (wdec) a -= p.wd * Yq[t * d];
                    }
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                if (s < mb && i16 == 0) p.deta[(size_t)bh * L + n0 + s] = wdec ? a - p.wd * wdw : a;
            }
            __syncthreads();
            // dP (into T2) and dV: through G's dependence on P and on v (and k)
            if (LN) {
                #pragma unroll
                for (int s = warp, it_ = 0; it_ < kRowIters; s += kWarps, ++it_) {
                    if (s >= mb) break;
                    const float *z = Pz + s * d;
                    const LnRow ln = ln_row(z, d, p.eps);
                    float gx[kMaxPerLane], Gv[kMaxPerLane], u[kMaxPerLane];
                    ln_grad_row(T3 + s * d, z, Kt + s * d, Vt + s * d, gam, bet, d, p.eps, p.ip != 0, ln, gx);
                    // T3 row s now holds G again (the same values as G); u = dG row
                    float su = 0.f, suG = 0.f, sxg = 0.f, sux = 0.f;
#pragma unroll
                    for (int i = 0; i < kMaxPerLane; ++i) {
                        const int j = lane + 32 * i;
                        u[i] = j < d ? dG[s * d + j] : 0.f;
                        Gv[i] = j < d ? G[s * d + j] : 0.f;
                        su += u[i];
                        suG += u[i] * Gv[i];
                        sxg += ln.xh[i] * gx[i];
                        sux += u[i] * ln.xh[i];
                    }
                    su = warp_sum(su);
                    suG = warp_sum(suG);
                    sxg = warp_sum(sxg);
                    sux = warp_sum(sux);
                    float f[kMaxPerLane], w[kMaxPerLane];
#pragma unroll
                    for (int i = 0; i < kMaxPerLane; ++i) {
                        const int j = lane + 32 * i;
                        const float a = (j < d && !p.ip) ? gam[j] * gam[j] : 0.f;
                        f[i] = ln.r * (a * u[i] - su * a / d - (u[i] * sxg + sux * (gx[i] + a * ln.xh[i])) / d);
                        w[i] = u[i];
                    }
                    ln_pi(f, ln.xh, d);
                    ln_pi(w, ln.xh, d);
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < kMaxPerLane; ++i) {
                        const int j = lane + 32 * i;
                        if (j >= d) continue;
                        const float wr = ln.r * w[i];
                        T2[s * d + j] = ln.r * f[i] - ln.r * suG * ln.xh[i] / d;   // dP
                        float dv;
                        if (p.ip) {
                            dv = -gam[j] * wr;
                            dgam_acc[i] = fmaf(-Vt[s * d + j], wr, dgam_acc[i]);
                            Vt[s * d + j] = 0.f;          // no dy term in dK
                        } else {
                            const float y = Vt[s * d + j] - Kt[s * d + j];
                            dv = -gam[j] * wr;            // dy
                            dgam_acc[i] = fmaf(2.f * gam[j] * ln.xh[i] + bet[j] - y, wr, dgam_acc[i]);
                            dbet_acc[i] = fmaf(gam[j], wr, dbet_acc[i]);
                            Vt[s * d + j] = dv;           // dy, for dK
                        }
                        store_io(dVg, s * d + j, dv);
                    }
                }
            } else {
                for (int i = tid; i < nt; i += kThreads) {
                    T2[i] = kf * dG[i];
                    store_io(dVg, i, -dG[i]);
                }
            }
            __syncthreads();
            // T3 <- G dW'^T again (the LN rows above overwrote it), T1 <- dP W^T
            if (LN) mm_xyt(T3, G, dW, mb, d, d);
            mm_xyt(T1, T2, W, mb, d, d);
            __syncthreads();
            // dK = dP W^T - E G dW'^T - E D^T Q (- dy with the residual LN)
            for (int tile = tid; tile < nt / 4; tile += kThreads) {
                const int s = tile / (d / 4), j = (tile - s * (d / 4)) * 4;
                const float4 t1 = f4(T1 + s * d + j), t3 = f4(T3 + s * d + j);
                float4 a = make_float4(t1.x - et[s] * t3.x, t1.y - et[s] * t3.y, t1.z - et[s] * t3.z,
                                       t1.w - et[s] * t3.w);
                if (LN) {
                    const float4 dy = f4(Vt + s * d + j);
                    a.x -= dy.x; a.y -= dy.y; a.z -= dy.z; a.w -= dy.w;
                }
#pragma unroll
                for (int t = 0; t < mb; ++t)
                    if (t >= s) fma4(a, -et[s] * Dm[t * mb + s], f4(Qt + t * d + j));
                store_io(dKg, s * d + j, a.x);
                store_io(dKg, s * d + j + 1, a.y);
                store_io(dKg, s * d + j + 2, a.z);
                store_io(dKg, s * d + j + 3, a.w);
            }
            // dW += Q^T dZbar + K^T dP;  dc += 1^T dZbar + 1^T dP
            {
                float esum = 0.f;
                if (wdec)
                    for (int s2 = 0; s2 < mb; ++s2) esum += et[s2];
                mm_xty_acc(dW, Qt, dZb, fq, 1.f, mb, d, d, 1.f - p.wd * esum);
            }
            __syncthreads();
            mm_xty_acc(dW, Kt, T2, nullptr, 1.f, mb, d, d);
            for (int j = tid; j < d; j += kThreads) {
                float a = 0.f;
#pragma unroll
                for (int s = 0; s < mb; ++s) a += dZb[s * d + j] + T2[s * d + j];
                dc[j] += a;
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < dd; i += kThreads) p.dW0[(size_t)bh * dd + i] = dW[i];
    for (int j = tid; j < d; j += kThreads) p.db0[(size_t)bh * d + j] = dc[j];
    if (LN) {
        // dgamma, dbeta of this row: the warps' accumulators summed in warp order
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int j = lane + 32 * i;
            if (j < d) {
                red[warp * 2 * d + j] = dgam_acc[i];
                red[warp * 2 * d + d + j] = dbet_acc[i];
            }
        }
        __syncthreads();
        for (int j = tid; j < 2 * d; j += kThreads) {
            float a = 0.f;
            for (int w = 0; w < kWarps; ++w) a += red[w * 2 * d + j];
            p.dgb[(size_t)bh * 2 * d + j] = a;
        }
    }
}

// out[h][e] = sum of part[i * stride + off + e] (e < n) over the call's rows i of head
// h = (hoff + i) mod H, in row order (deterministic); heads without a row get 0
__global__ void sum_over_rows_kernel(const float *part, float *out, int rows, int H, int hoff, int stride, int n,
                                     int off)
{
    const size_t total = (size_t)H * n;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int hh = (int)(i / n);
        const size_t e = i - (size_t)hh * n;
        const int first = ((hh - hoff) % H + H) % H;   // the first row of head hh
        float a = 0.f;
        for (int r = first; r < rows; r += H) a += part[(size_t)r * stride + off + e];
        out[i] = a;
    }
}

constexpr size_t kMaxSmem = 227 * 1024;

// bytes of the prefetch buffer (four mb x d tiles of I/O elements and mb floats of eta), used
// by the kernel specialised for d = 64, b = 16
size_t prefetch_bytes(const ttt_desc &s)
{
    if (!(s.d == 64 && s.mini_batch == 16)) return 0;
    const size_t es = s.io_dtype == TTT_BF16 ? 2 : 4;
    return 4 * (size_t)s.mini_batch * s.d * es + (size_t)s.mini_batch * 4;
}

size_t smem_for(const ttt_desc &s, int ck)
{
    // states, dW and dc, nine mb x d tiles, the small block; with LN or weight decay P, Zbar,
    // gamma, beta and Q W; with LN and d < 16 the dgamma/dbeta reduction's own area
    const size_t d = s.d, mb = s.mini_batch, states = ck * (d * d + d);
    const size_t red = 2 * d * (kThreads / 32);
    const bool wd = s.weight_decay != 0.f;
    size_t n = states + d * d + d + 9 * mb * d + small_floats((int)mb);
    if (s.residual_ln || wd) n += 2 * mb * d + 2 * d;   // P, Zbar / dZbar, gamma, beta
    if (wd) n += mb * d;                                // Q W
    if (s.residual_ln && red > states) n += red;
    n = (n + 3) & ~(size_t)3;   // the prefetch buffer starts 16-byte aligned
    return n * sizeof(float) + prefetch_bytes(s);
}

}  // namespace

int linear_bwd_checkpoint_every(const ttt_desc &s)
{
    if (s.d > 128 || s.d % 4 != 0 || s.mini_batch > 64) return 0;
    for (int ck : {4, 2, 1})
        if (smem_for(s, ck) <= kMaxSmem) return ck;
    return 0;
}

size_t linear_bwd_workspace_bytes(const ttt_desc &s)
{
    const int ck = linear_bwd_checkpoint_every(s);
    if (!ck) return 0;
    const size_t rows = call_rows(s), d = s.d;
    const size_t nmb = s.L / s.mini_batch, nck = (nmb + ck - 1) / ck;
    size_t bytes = rows * nck * (d * d + d) * sizeof(float);
    if (!s.init_per_batch) bytes += rows * (d * d + d) * sizeof(float);   // per-(batch, head) partials
    if (s.residual_ln) bytes += rows * 2 * d * sizeof(float);              // dgamma, dbeta partials
    return (bytes + 255) / 256 * 256;
}

cudaError_t launch_linear_bwd(const LinearBwdArgs &a)
{
    const ttt_desc &s = a.desc;
    const int ck = linear_bwd_checkpoint_every(s);
    const int rows = call_rows(s);
    const size_t d = s.d, nmb = s.L / s.mini_batch, nck = (nmb + ck - 1) / ck;
    float *ckpt = static_cast<float *>(a.workspace);
    float *part = ckpt + (size_t)rows * nck * (d * d + d);
    float *dgb = part + (s.init_per_batch ? 0 : (size_t)rows * (d * d + d));
    BwdParams p{s.H, s.L, s.d, s.mini_batch, ck, s.init_per_batch, s.loss == TTT_LOSS_INNER_PRODUCT,
                s.ln_eps, s.weight_decay, a.Q, a.K, a.V, a.dZ, a.eta, a.W0, a.b0, a.gamma, a.beta, a.dW_final, a.db_final,
                a.dQ, a.dK, a.dV, a.deta, s.init_per_batch ? a.dW0 : part,
                s.init_per_batch ? a.db0 : part + (size_t)rows * d * d, dgb, ckpt, head_offset(s)};
    const size_t smem = smem_for(s, ck);
    p.pf_off = (int)((smem - prefetch_bytes(s)) / sizeof(float));
    const bool f32 = s.io_dtype == TTT_F32, ln = s.residual_ln != 0, fixed = s.d == 64 && s.mini_batch == 16;
    const void *k;
    if (fixed)
        k = f32 ? (ln ? (const void *)linear_bwd_kernel<float, true, 64, 16> : (const void *)linear_bwd_kernel<float, false, 64, 16>)
                : (ln ? (const void *)linear_bwd_kernel<__nv_bfloat16, true, 64, 16>
                      : (const void *)linear_bwd_kernel<__nv_bfloat16, false, 64, 16>);
    else
        k = f32 ? (ln ? (const void *)linear_bwd_kernel<float, true, 0, 0> : (const void *)linear_bwd_kernel<float, false, 0, 0>)
                : (ln ? (const void *)linear_bwd_kernel<__nv_bfloat16, true, 0, 0>
                      : (const void *)linear_bwd_kernel<__nv_bfloat16, false, 0, 0>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {&p};
    e = cudaLaunchKernel(k, dim3(rows), dim3(kThreads), args, smem, a.stream);
    if (e != cudaSuccess) return e;
    if (ln) {   // dgamma, dbeta [H, d]: per-head sums of the rows' partials ([rows][dgamma | dbeta])
        sum_over_rows_kernel<<<148, 256, 0, a.stream>>>(dgb, a.dgamma, rows, s.H, head_offset(s), (int)(2 * d),
                                                       (int)d, 0);
        sum_over_rows_kernel<<<148, 256, 0, a.stream>>>(dgb, a.dbeta, rows, s.H, head_offset(s), (int)(2 * d),
                                                       (int)d, (int)d);
        if ((e = cudaGetLastError()) != cudaSuccess || s.init_per_batch) return e;
    } else if (s.init_per_batch) {
        return e;
    }
    // head-shared initial state: sum the per-(batch, head) gradients over the call's rows
    sum_over_rows_kernel<<<148, 256, 0, a.stream>>>(part, a.dW0, rows, s.H, head_offset(s), (int)(d * d),
                                                   (int)(d * d), 0);
    sum_over_rows_kernel<<<148, 256, 0, a.stream>>>(part + (size_t)rows * d * d, a.db0, rows, s.H,
                                                   head_offset(s), (int)d, (int)d, 0);
    return cudaGetLastError();
}

}  // namespace ttt
