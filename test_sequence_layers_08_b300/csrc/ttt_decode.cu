// ttt_decode.cu -- TTT-Linear decode: the tokens of a call are processed one at a time
// (mini-batch size 1) from a fast-weight state (W, c) that lives in device memory between
// calls and is updated in place.
//
// Per token t of every (batch, head) -- the update/apply recurrence of the damodev.csdn.net
// TTT article, section 3.1 (the output reads the weights after the token's own update), with
// mini-batch size 1 of sections 4.1-4.2 and the residual LayerNorm of the lryc.cn article,
// section 2.1:
//   z = k_t W + c
//   g = z - v_t                      (plain)   or   g = LNbwd(z; v_t - k_t)   (residual LN)
//   W -= eta_t k_t^T g,   c -= eta_t g
//   o = q_t W + c,   Z_t = o   or   Z_t = q_t + LN(o)
// With the residual LayerNorm the output is taken from the products with the state before
// the update, o = q_t W_old + c_new - eta_t (q_t . k_t) g  ((1 - eta_t lambda) q_t W_old with
// decay), so one sweep over W gives both k_t W_old and q_t W_old and a token costs two
// sweeps (products, update) instead of three; the q . k butterfly hides under the
// LayerNorm's.  Without the LayerNorm the chain per token is short and three sweeps with
// more independent partial sums are faster (B300: 17.2 against 18.1 us for 16 tokens).
// with LNbwd the gradient of 1/2 |gamma xhat + beta - y|^2, xhat = (z - mu) r, through the
// LayerNorm: g = r (gx - mean(gx) - xhat mean(gx xhat)), gx = gamma (gamma xhat + beta - y).
// The inner-learner variants of the ai-feeds Modular TTT page: with the inner-product loss
// -<f(k), v>, g = -v (plain) or the LayerNorm backward of the upstream -v (gx = -gamma v);
// with weight decay lambda the update is W <- (1 - eta_t lambda) W - eta_t k_t^T g (the bias
// is not decayed).
//
// B300 design.  A decode step is a chain of 64 x 64 matrix-vector products on a 16 KB state
// per (batch, head): latency- and launch-bound work that suits FP32 FMA, not tensor cores.
//   * one warp per (batch, head), four per CTA (one per SM sub-partition);
//   * lane j holds columns 2j, 2j + 1 of W (128 registers) for all the call's tokens: W is
//     read and written once per call;
//   * each token's q and k rows are staged in a per-warp shared-memory row, so every lane
//     reads k_i and q_i as 16-byte broadcasts;
//   * sums over the 64 features are warp butterflies; the LayerNorm statistics take two
//     passes (the mean, then the centred second moment).
// Without the LayerNorm the columns of the state never mix (column j of W and c evolves from
// column j of k W + c and of v alone), so a (batch, head) is split over four warps of 16
// columns each: lane l owns column 16 w + (l mod 16) and rows 32 (l / 16) .. + 31 of it (32
// registers), a token costs three 32-long sweeps and one shuffle per product, and the
// warps of a head need no communication.  Tokens are staged eight at a time (q, k rows in
// shared memory, v and eta in registers) while the next eight are loaded, so the short
// per-token chain does not wait on a global load round trip per token.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int D = 64;
constexpr int kWarps = 4;

struct DecodeParams {
    int BH, H, T, hoff;
    float eps;
    int ip;       // inner-product loss
    float wd;     // weight decay lambda
    const void *Q, *K, *V;
    const float *eta;
    float *W, *b;
    const float *gamma, *beta;
    void *Z;
};

template <bool BF16>
__device__ __forceinline__ float2 load_pair(const void *base, size_t idx)   // elements idx, idx + 1
{
    if (BF16) {
        const uint32_t u = reinterpret_cast<const uint32_t *>(base)[idx >> 1];
        return make_float2(ptx::bf16_lo(u), ptx::bf16_hi(u));
    }
    return reinterpret_cast<const float2 *>(base)[idx >> 1];
}

template <bool BF16>
__device__ __forceinline__ void store_pair(void *base, size_t idx, float x, float y)
{
    if (BF16)
        reinterpret_cast<uint32_t *>(base)[idx >> 1] = ptx::pack_bf16(x, y);
    else
        reinterpret_cast<float2 *>(base)[idx >> 1] = make_float2(x, y);
}

__device__ __forceinline__ float warp_sum(float a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    return a;
}

__device__ __forceinline__ float2 warp_sum2(float a, float b)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    return make_float2(a, b);
}

__device__ __forceinline__ float3 warp_sum3(float a, float b, float c)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
        c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    return make_float3(a, b, c);
}

template <bool BF16, bool LN, bool WD>
__global__ void __launch_bounds__(kWarps * 32)
linear_decode_kernel(DecodeParams p)
{
    __shared__ float4 rows[kWarps][2][D / 4];   // per warp: q and k of the current token
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x * kWarps + warp;
    if (bh >= p.BH) return;   // whole warps leave; the kernel uses no block-wide barrier
    const int h = (p.hoff + bh) % p.H;
    const int j0 = 2 * lane;  // this lane's two features / columns of W

    float w[D][2];
    float *Wg = p.W + (size_t)bh * D * D;
#pragma unroll
    for (int i = 0; i < D; ++i) {
        const float2 v = *reinterpret_cast<const float2 *>(Wg + i * D + j0);
        w[i][0] = v.x;
        w[i][1] = v.y;
    }
    float *bg = p.b + (size_t)bh * D;
    float c0 = bg[j0], c1 = bg[j0 + 1];
    float ga0 = 1.f, ga1 = 1.f, be0 = 0.f, be1 = 0.f;
    if (LN) {
        ga0 = p.gamma[(size_t)h * D + j0];
        ga1 = p.gamma[(size_t)h * D + j0 + 1];
        be0 = p.beta[(size_t)h * D + j0];
        be1 = p.beta[(size_t)h * D + j0 + 1];
    }
    float *qs = reinterpret_cast<float *>(rows[warp][0]);
    float *ks = reinterpret_cast<float *>(rows[warp][1]);

    // x W for the row staged at xs (16-byte broadcasts), as four partial sums per column
    auto row_times_w = [&](const float4 *xs, float &r0, float &r1) {
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i4 = 0; i4 < D / 4; ++i4) {
            const float4 x = xs[i4];
            const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                a0[e] = fmaf(xv[e], w[4 * i4 + e][0], a0[e]);
                a1[e] = fmaf(xv[e], w[4 * i4 + e][1], a1[e]);
            }
        }
        r0 = (a0[0] + a0[1]) + (a0[2] + a0[3]);
        r1 = (a1[0] + a1[1]) + (a1[2] + a1[3]);
    };
    // k W and q W for the rows staged at ks4, qs4 (16-byte broadcasts), four partial sums each
    auto rows_times_w = [&](const float4 *ks4, const float4 *qs4, float &z0, float &z1, float &y0,
                            float &y1) {
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
        float b0[4] = {0.f, 0.f, 0.f, 0.f}, b1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i4 = 0; i4 < D / 4; ++i4) {
            const float4 x = ks4[i4], y = qs4[i4];
            const float xv[4] = {x.x, x.y, x.z, x.w}, yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                a0[e] = fmaf(xv[e], w[4 * i4 + e][0], a0[e]);
                a1[e] = fmaf(xv[e], w[4 * i4 + e][1], a1[e]);
                b0[e] = fmaf(yv[e], w[4 * i4 + e][0], b0[e]);
                b1[e] = fmaf(yv[e], w[4 * i4 + e][1], b1[e]);
            }
        }
        z0 = (a0[0] + a0[1]) + (a0[2] + a0[3]);
        z1 = (a1[0] + a1[1]) + (a1[2] + a1[3]);
        y0 = (b0[0] + b0[1]) + (b0[2] + b0[3]);
        y1 = (b1[0] + b1[1]) + (b1[2] + b1[3]);
    };

    // the next token's inputs are loaded while the current one is computed
    const size_t row0 = (size_t)bh * p.T;
    float2 qn = load_pair<BF16>(p.Q, row0 * D + j0), kn = load_pair<BF16>(p.K, row0 * D + j0),
           vn = load_pair<BF16>(p.V, row0 * D + j0);
    float en = p.eta[row0];
    for (int t = 0; t < p.T; ++t) {
        const size_t base = (row0 + t) * D + j0;
        const float2 q = qn, k = kn, v = vn;
        const float et = en;
        if (t + 1 < p.T) {
            qn = load_pair<BF16>(p.Q, base + D);
            kn = load_pair<BF16>(p.K, base + D);
            vn = load_pair<BF16>(p.V, base + D);
            en = p.eta[row0 + t + 1];
        }
        *reinterpret_cast<float2 *>(qs + j0) = q;
        *reinterpret_cast<float2 *>(ks + j0) = k;
        __syncwarp();

        // key-side product with the state before this token's update (with the LayerNorm also
        // the query-side product and q . k)
        float z0, z1, y0 = 0.f, y1 = 0.f, qk = 0.f;
        if (LN)
            rows_times_w(rows[warp][1], rows[warp][0], z0, z1, y0, y1);
        else
            row_times_w(rows[warp][1], z0, z1);
        z0 += c0;
        z1 += c1;
        float g0, g1;
        if (LN) {
            // one reduction round for q . k and the sums of z - z_0 and (z - z_0)^2, z_0 this
            // token's first feature: shifted one-pass sums, free of cancellation when z has a
            // common offset much larger than its spread, and depending on this token alone
            const float sh = __shfl_sync(0xffffffffu, z0, 0);
            const float d0 = z0 - sh, d1 = z1 - sh;
            const float3 s3 = warp_sum3(fmaf(q.x, k.x, q.y * k.y), d0 + d1, fmaf(d0, d0, d1 * d1));
            qk = s3.x;
            const float md = s3.y * (1.f / D), mu = sh + md;
            const float zc0 = z0 - mu, zc1 = z1 - mu;
            const float r = rsqrtf(fmaxf(s3.z * (1.f / D) - md * md, 0.f) + p.eps);
            const float xh0 = zc0 * r, xh1 = zc1 * r;
            const float gx0 = p.ip ? -ga0 * v.x : ga0 * (fmaf(ga0, xh0, be0) - (v.x - k.x));
            const float gx1 = p.ip ? -ga1 * v.y : ga1 * (fmaf(ga1, xh1, be1) - (v.y - k.y));
            const float2 m = warp_sum2(gx0 + gx1, fmaf(gx0, xh0, gx1 * xh1));
            const float m1 = m.x * (1.f / D), m2 = m.y * (1.f / D);
            g0 = r * (gx0 - m1 - xh0 * m2);
            g1 = r * (gx1 - m1 - xh1 * m2);
        } else {
            g0 = p.ip ? -v.x : z0 - v.x;
            g1 = p.ip ? -v.y : z1 - v.y;
        }

        // W <- (1 - eta lambda) W - eta k^T g,  c -= eta g   (the factor is 1 without decay)
        const float eg0 = et * g0, eg1 = et * g1;
        const float dec = WD ? 1.f - et * p.wd : 1.f;
#pragma unroll
        for (int i4 = 0; i4 < D / 4; ++i4) {
            const float4 x = rows[warp][1][i4];
            w[4 * i4][0] = fmaf(-eg0, x.x, WD ? dec * w[4 * i4][0] : w[4 * i4][0]);
            w[4 * i4][1] = fmaf(-eg1, x.x, WD ? dec * w[4 * i4][1] : w[4 * i4][1]);
            w[4 * i4 + 1][0] = fmaf(-eg0, x.y, WD ? dec * w[4 * i4 + 1][0] : w[4 * i4 + 1][0]);
            w[4 * i4 + 1][1] = fmaf(-eg1, x.y, WD ? dec * w[4 * i4 + 1][1] : w[4 * i4 + 1][1]);
            w[4 * i4 + 2][0] = fmaf(-eg0, x.z, WD ? dec * w[4 * i4 + 2][0] : w[4 * i4 + 2][0]);
            w[4 * i4 + 2][1] = fmaf(-eg1, x.z, WD ? dec * w[4 * i4 + 2][1] : w[4 * i4 + 2][1]);
            w[4 * i4 + 3][0] = fmaf(-eg0, x.w, WD ? dec * w[4 * i4 + 3][0] : w[4 * i4 + 3][0]);
            w[4 * i4 + 3][1] = fmaf(-eg1, x.w, WD ? dec * w[4 * i4 + 3][1] : w[4 * i4 + 3][1]);
        }
        c0 -= eg0;
        c1 -= eg1;

        // the output with the weights after this token's update
        float o0, o1;
        if (LN) {   // q W_new + c_new = dec (q W_old) - eta (q . k) g + c_new
            o0 = fmaf(-eg0, qk, fmaf(dec, y0, c0));
            o1 = fmaf(-eg1, qk, fmaf(dec, y1, c1));
        } else {
            row_times_w(rows[warp][0], o0, o1);
            o0 += c0;
            o1 += c1;
        }
        if (LN) {   // shifted one-pass sums of o, as for z
            const float sh = __shfl_sync(0xffffffffu, o0, 0);
            const float d0 = o0 - sh, d1 = o1 - sh;
            const float2 s2 = warp_sum2(d0 + d1, fmaf(d0, d0, d1 * d1));
            const float md = s2.x * (1.f / D), mu = sh + md;
            const float oc0 = o0 - mu, oc1 = o1 - mu;
            const float r = rsqrtf(fmaxf(s2.y * (1.f / D) - md * md, 0.f) + p.eps);
            o0 = q.x + fmaf(ga0 * oc0, r, be0);
            o1 = q.y + fmaf(ga1 * oc1, r, be1);
        }
        store_pair<BF16>(p.Z, base, o0, o1);
        __syncwarp();   // every lane is done with the staged rows before the next token
    }

#pragma unroll
    for (int i = 0; i < D; ++i) *reinterpret_cast<float2 *>(Wg + i * D + j0) = make_float2(w[i][0], w[i][1]);
    bg[j0] = c0;
    bg[j0 + 1] = c1;
}

constexpr int kColWarps = 4;                    // warps per (batch, head) without the LayerNorm
constexpr int kColsPerWarp = D / kColWarps;     // 16: lanes l and l + 16 share a column
constexpr int kRowPad = 4;                      // the staged rows' second half starts 16 bytes late

template <bool BF16>
__device__ __forceinline__ float load_one(const void *base, size_t idx)
{
    if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
    return reinterpret_cast<const float *>(base)[idx];
}

template <bool BF16>
__device__ __forceinline__ void store_one(void *base, size_t idx, float x)
{
    if (BF16)
        reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float *>(base)[idx] = x;
}

constexpr int kTokBlock = 8;                    // tokens staged per block (the next block is loaded meanwhile)

// Decode without the residual LayerNorm, a (batch, head) over kColWarps warps by column.
template <bool BF16, bool WD>
__global__ void __launch_bounds__(kWarps * 32)
linear_decode_cols_kernel(DecodeParams p)
{
    // per warp and staged token: q and k, features 32..63 placed kRowPad floats late so that
    // the two half-warps' 16-byte broadcasts fall in different banks
    __shared__ __align__(16) float rows[kWarps][kTokBlock][2][D + kRowPad];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + warp;
    const int bh = gw / kColWarps, part = gw - bh * kColWarps;
    if (bh >= p.BH) return;   // whole warps leave; the kernel uses no block-wide barrier
    const int col = part * kColsPerWarp + (lane & 15), r0 = (lane >> 4) * 32;
    const int off = (lane >> 4) * (32 + kRowPad);   // this half's rows in a staged row
    const int j0 = 2 * lane;                        // the pair of features this lane stages
    const int sp = j0 < 32 ? j0 : j0 + kRowPad;     // staged position of feature j0

    float w[32];
    float *Wg = p.W + (size_t)bh * D * D;
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = Wg[(r0 + i) * D + col];
    float *bg = p.b + (size_t)bh * D;
    float c = bg[col];

    // this half's partial of x W[:, col] for the staged row xs (four partial sums), completed
    // with the other half's through one shuffle
    auto half_dot = [&](const float *xs) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xs + off);
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
            const float4 x = x4[i4];
            a[0] = fmaf(x.x, w[4 * i4], a[0]);
            a[1] = fmaf(x.y, w[4 * i4 + 1], a[1]);
            a[2] = fmaf(x.z, w[4 * i4 + 2], a[2]);
            a[3] = fmaf(x.w, w[4 * i4 + 3], a[3]);
        }
        const float part_sum = (a[0] + a[1]) + (a[2] + a[3]);
        return part_sum + __shfl_xor_sync(0xffffffffu, part_sum, 16);
    };

    // a block of tokens in registers: this lane's pairs of q and k, v of its column, eta
    const size_t row0 = (size_t)bh * p.T;
    float2 qn[kTokBlock], kn[kTokBlock];
    float vn[kTokBlock], en[kTokBlock];
    auto fetch = [&](int t0) {
#pragma unroll
        for (int u = 0; u < kTokBlock; ++u)
            if (t0 + u < p.T) {
                const size_t base = (row0 + t0 + u) * D;
                qn[u] = load_pair<BF16>(p.Q, base + j0);
                kn[u] = load_pair<BF16>(p.K, base + j0);
                vn[u] = load_one<BF16>(p.V, base + col);
                en[u] = p.eta[row0 + t0 + u];
            }
    };
    fetch(0);
    for (int t0 = 0; t0 < p.T; t0 += kTokBlock) {
        float vb[kTokBlock], eb[kTokBlock];
#pragma unroll
        for (int u = 0; u < kTokBlock; ++u) {
            if (t0 + u < p.T) {
                *reinterpret_cast<float2 *>(&rows[warp][u][0][sp]) = qn[u];
                *reinterpret_cast<float2 *>(&rows[warp][u][1][sp]) = kn[u];
            }
            vb[u] = vn[u];
            eb[u] = en[u];
        }
        __syncwarp();
        if (t0 + kTokBlock < p.T) fetch(t0 + kTokBlock);   // the next block, while this one runs
#pragma unroll
        for (int u = 0; u < kTokBlock; ++u) {
            if (t0 + u >= p.T) break;
            const float *qs = rows[warp][u][0], *ks = rows[warp][u][1];
            const float z = half_dot(ks) + c;
            const float g = p.ip ? -vb[u] : z - vb[u];
            // W[:, col] <- (1 - eta lambda) W[:, col] - eta k^T g,  c -= eta g
            const float eg = eb[u] * g;
            const float dec = WD ? 1.f - eb[u] * p.wd : 1.f;
            const float4 *k4 = reinterpret_cast<const float4 *>(ks + off);
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
                const float4 x = k4[i4];
                w[4 * i4] = fmaf(-eg, x.x, WD ? dec * w[4 * i4] : w[4 * i4]);
                w[4 * i4 + 1] = fmaf(-eg, x.y, WD ? dec * w[4 * i4 + 1] : w[4 * i4 + 1]);
                w[4 * i4 + 2] = fmaf(-eg, x.z, WD ? dec * w[4 * i4 + 2] : w[4 * i4 + 2]);
                w[4 * i4 + 3] = fmaf(-eg, x.w, WD ? dec * w[4 * i4 + 3] : w[4 * i4 + 3]);
            }
            c -= eg;
            // the output with the weights after this token's update
            const float o = half_dot(qs) + c;
            if (lane < 16) store_one<BF16>(p.Z, (row0 + t0 + u) * D + col, o);
        }
        __syncwarp();   // every lane is done with the staged rows before the next block
    }

#pragma unroll
    for (int i = 0; i < 32; ++i) Wg[(r0 + i) * D + col] = w[i];
    if (lane < 16) bg[col] = c;
}

}  // namespace

bool linear_decode_supported(const ttt_desc &d) { return d.d == D && d.mini_batch == 1; }

cudaError_t launch_linear_decode(const DecodeArgs &a)
{
    const ttt_desc &d = a.desc;
    const int BH = call_rows(d);
    DecodeParams p{BH, d.H, d.L, head_offset(d), d.ln_eps, d.loss == TTT_LOSS_INNER_PRODUCT,
                   d.weight_decay, a.Q, a.K, a.V, a.eta, a.W, a.b, a.gamma, a.beta, a.Z};
    const int grid = (BH + kWarps - 1) / kWarps;
    const bool bf16 = d.io_dtype == TTT_BF16, ln = d.residual_ln != 0, wd = d.weight_decay != 0.f;
    using K = void (*)(DecodeParams);
    if (!ln) {   // split by column: kColWarps warps per (batch, head)
        const K cols[2][2] = {{linear_decode_cols_kernel<false, false>, linear_decode_cols_kernel<false, true>},
                              {linear_decode_cols_kernel<true, false>, linear_decode_cols_kernel<true, true>}};
        const int cgrid = (int)(((long long)BH * kColWarps + kWarps - 1) / kWarps);
        cols[bf16][wd]<<<cgrid, kWarps * 32, 0, a.stream>>>(p);
        return cudaGetLastError();
    }
    const K table[2][2][2] = {{{linear_decode_kernel<false, false, false>, linear_decode_kernel<false, false, true>},
                               {linear_decode_kernel<false, true, false>, linear_decode_kernel<false, true, true>}},
                              {{linear_decode_kernel<true, false, false>, linear_decode_kernel<true, false, true>},
                               {linear_decode_kernel<true, true, false>, linear_decode_kernel<true, true, true>}}};
    table[bf16][ln][wd]<<<grid, kWarps * 32, 0, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ttt
