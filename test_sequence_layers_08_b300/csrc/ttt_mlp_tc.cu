// ttt_mlp_tc.cu -- fused TTT-MLP forward for bf16 I/O, d = 64, d_hidden = 256, b = 16.
//
// The method (TTT-MLP of the lryc.cn TTT article, section 2.1: f(x) = x + LN(f_res(x)),
// f_res = GELU(x W1 + b1) W2 + b2; mini-batch gradient descent of the damodev.csdn.net
// TTT article, sections 4.1-4.2, every gradient of a mini-batch taken at its starting
// weights).  Per (batch, head) and mini-batch n (16 tokens):
//   Z1 = K W1 + b1,  X2 = GELU(Z1),  Z2 = X2 W2 + b2
//   G2 = LNbwd(Z2; V - K)  (or Z2 - V),   G1 = (G2 W2^T) . GELU'(Z1)
//   W1 -= K^T diag(eta) G1,  b1 -= eta^T G1,  W2 -= X2^T diag(eta) G2,  b2 -= eta^T G2
// and the outputs, read with the weights after each token's own update (dual form):
//   Zb1 = Q W1 + b1 - (eta_s (Q_t . K_s + 1) [s <= t]) G1,   Xb2 = GELU(Zb1)
//   Zb2 = Xb2 W2 + b2 - (eta_s (Xb2_t . X2_s + 1) [s <= t]) G2,   Z = Q + LN(Zb2)
// with the weights of the mini-batch start on the right-hand sides.
//
// B300 design.  One CTA per (batch, head), eight warps: two per SM sub-partition, so each
// thread may hold 255 registers (two warps fill a sub-partition's register file) and the
// fp32 weight slices plus the step's temporaries fit without spilling:
//   * 64-token stages of Q, K, V (TMA, 128-byte swizzle) and eta stream into a 4-deep
//     shared-memory ring; thread 0 refills a slot once no warp reads it any more;
//   * warps 0-7 each own 32 of the 256 hidden units: their rows of W1^T and of W2 stay in
//     registers as fp32 warp-MMA accumulators for the whole scan.  Every contraction is a
//     bf16 m16n8k16 warp MMA.  Contractions inside a warp's hidden slice (Z1, Q W1, G1,
//     both updates, the first output correction) read only registers and the stage tiles;
//     the two contractions over all 256 hidden units (X2 W2, Xb2 W2) and the 16 x 16
//     Gram Xb2 X2^T read bf16 copies of X2, Xb2 and W2 that every warp writes into shared
//     memory for its slice;
//   * warps 0-3 also own 16 of the 64 outputs each and run both LayerNorms (statistics in
//     fp32: warp reduce-scatter plus one shared-memory exchange);
//   * the two contractions over all hidden units are split by hidden half: warps w and
//     w + 4 take units 0-127 and 128-255 for the outputs of warp w, and warps 4-7 hand
//     their fp32 partials over through shared memory; the 16 x 16 Gram Xb2 X2^T is split
//     the same way over warps 4-7.
// Per mini-batch all eight warps meet at five named barriers (warps 4-7 run into the next
// mini-batch's first layer while warps 0-3 finish the output); every mbarrier wait is bounded.
// Inner-learner variants (ai-feeds Modular TTT page): the inner-product loss -<f(k), v> zeroes
// the gamma^2, beta and k coefficients of the LayerNorm backward (G2 = -V without it); weight
// decay (a template switch) scales W1, W2 by 1 - lambda S before their updates and the
// query-side products of both layers by 1 - lambda cum_t around the bias.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int D = 64;           // model / head dim
constexpr int DH = 256;         // hidden dim
constexpr int MB = 16;          // mini-batch
constexpr int ST = 64;          // tokens per pipeline stage
constexpr int TPS = ST / MB;    // mini-batches per stage
constexpr int NSS = 4;          // stages in the ring
constexpr int kCompute = 8;     // compute warps
constexpr int kThreads = kCompute * 32;
constexpr uint32_t kStageTileBytes = ST * D * 2;   // 8 KB

struct __align__(1024) Smem {
    __nv_bfloat16 q[NSS][ST * D];       // 128-byte swizzled rows of 64 features
    __nv_bfloat16 k[NSS][ST * D];
    __nv_bfloat16 v[NSS][ST * D];
    __nv_bfloat16 w2b[DH * D];          // W2 [h][o] at the mini-batch start, 128-byte swizzle
    __nv_bfloat16 x2[MB * DH];          // X2 [t][h], 512-byte rows, 16-byte chunks XOR (t & 7)
    __nv_bfloat16 xb2[MB * DH];         // Xb2 [t][h], same layout
    __nv_bfloat16 g2[MB * D];           // G2 [t][o], 128-byte swizzle
    __nv_bfloat16 eg2[MB * D];          // -eta G2 [t][o], 128-byte swizzle
    __nv_bfloat16 zst[MB * D];          // Z staging [t][o], 128-byte swizzle
    float eta[NSS][ST];
    uint32_t a1f[2][32][2];             // eta_s (Q_t . K_s + 1) [s <= t] as B fragments [s half][lane][t n-tile]
    float parta2[2][2][32][4];          // Xb2_t . X2_s partials [s half][hidden half][lane][4] (warps 4-7)
    float part2[4][32][8];              // X W2 partials over hidden units 128-255 [output warp][lane][8]
    // LayerNorm exchange tables [parity][token][quantity * 4 + warp]; rows padded (36, 12
    // floats) so the 16-byte reads are free of bank conflicts
    float red[2][MB][36];               // six backward sums
    float zred[2][MB][12];              // output sums: z, z^2
    unsigned long long full[NSS];
    int abort_flag;
};

static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory budget");

struct Params {
    int H, L, N, NST, init_per_batch;
    float eps;
    long long wait_ns;
    int withhold_loads;
    const float *eta, *W1, *b1, *W2, *b2, *gamma, *beta;
    float *W1f, *b1f, *W2f, *b2f;
    unsigned int *status;
    int hoff;                // head index of row 0 of this call
    int ip;                  // inner-product loss
    float wd;                // weight decay lambda (the WD instantiation)
};

constexpr long long kDrainNs = 1000000000ll;

// Barrier ids: 1 = the eight compute warps, 2 = the four LayerNorm warps.
constexpr int kBarAll = 1, kBarLn = 2;

__device__ __noinline__ bool mlp_wait_slow(uint32_t bar, uint32_t parity, long long limit, int *abort_flag,
                                           unsigned int *status)
{
    if (*(volatile int *)abort_flag) return false;
    if (ptx::mbar_wait_bounded(bar, parity, limit)) return true;
    *(volatile int *)abort_flag = 1;
    atomicOr(status, kStatusTimeout);
    return false;
}

// X2 / Xb2 tile: row t (token), 16-byte chunk ch (8 hidden units)
__device__ __forceinline__ uint32_t xh_off(int t, int ch) { return (uint32_t)(t * 512 + ((ch ^ (t & 7)) << 4)); }

// GELU(tanh): GELU(x) = x p with p = 1/2 (1 + tanh u), u = sqrt(2/pi) (x + 0.044715 x^3), and
// GELU'(x) = p + 1/2 x (1 - tanh(u)^2) du/dx.  tanh is the PTX approximate instruction (one
// MUFU operation per value; its relative error, about 2^-11, is far below the bf16 rounding
// of every GELU value, which becomes an MMA operand right after).
__device__ __forceinline__ float tanh_fast(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kGs = 0.7978845608028654f;   // sqrt(2/pi)
constexpr float kGa = 0.044715f;
__device__ __forceinline__ float gelu(float x)
{
    const float h = 0.5f * x;
    return fmaf(h, tanh_fast(kGs * x * fmaf(kGa, x * x, 1.f)), h);
}
__device__ __forceinline__ void gelu_and_prime(float x, float &y, float &dy)
{
    const float x2 = x * x, h = 0.5f * x;
    const float th = tanh_fast(kGs * x * fmaf(kGa, x2, 1.f));
    y = fmaf(h, th, h);
    // du/dx = sqrt(2/pi) (1 + 3 a x^2)
    const float du = fmaf(3.f * kGs * kGa, x2, kGs);
    dy = fmaf(h * du, fmaf(-th, th, 1.f), fmaf(0.5f, th, 0.5f));
}

template <bool LN, bool WD>
__global__ void __maxnreg__(255)
mlp_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, Params p, __nv_bfloat16 *Zg)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    Smem &s = *reinterpret_cast<Smem *>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, h = (p.hoff + bh) % p.H;
    const int N = p.N;

    // stage st -> ring slot st % NSS (thread 0 only)
    const float *eta_bh = p.eta + (size_t)bh * p.L;
    auto issue_stage = [&](int st) {
        const int b = st % NSS, ntok = min(ST, p.L - st * ST);
        const uint32_t fb = ptx::smem_addr(&s.full[b]);
        ptx::mbar_arrive_expect_tx(fb, 3 * kStageTileBytes + ntok * 4);
        ptx::tma_load_3d(ptx::smem_addr(s.q[b]), &tmQ, fb, 0, st * ST, bh);
        ptx::tma_load_3d(ptx::smem_addr(s.k[b]), &tmK, fb, 0, st * ST, bh);
        ptx::tma_load_3d(ptx::smem_addr(s.v[b]), &tmV, fb, 0, st * ST, bh);
        ptx::bulk_load(ptx::smem_addr(s.eta[b]), eta_bh + st * ST, ntok * 4, fb);
    };
    const int nissue = p.withhold_loads ? 0 : p.NST;
    int issued = 0;   // stages handed to the copy engine (thread 0)
    if (tid == 0) {
        for (int i = 0; i < NSS; ++i) ptx::mbar_init(ptx::smem_addr(&s.full[i]), 1);
        s.abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        for (; issued < min(NSS, nissue); ++issued) issue_stage(issued);
    }
    __syncthreads();

    // ------------------------------------------------------------------ compute warps
    const int g = lane >> 2, c = lane & 3, mrow = lane & 7, mat = lane >> 3;
    const int hb = warp * 32;                  // first hidden unit of this warp
    const bool lnw = warp < 4;                 // LayerNorm / output warp
    const int o0 = warp * 16 + g, o1 = o0 + 8; // its two outputs (warps 0-3)
    bool aborted = false;
    auto wait_stage = [&](int st) {
        if (aborted) return;
        const uint32_t bar = ptx::smem_addr(&s.full[st % NSS]);
        if (ptx::mbar_try_wait(bar, (st / NSS) & 1)) return;
        aborted = !mlp_wait_slow(bar, (st / NSS) & 1, p.wait_ns, &s.abort_flag, p.status);
    };
    auto tile_addr = [&](const __nv_bfloat16 (*arr)[ST * D], int n, int t, int chunk) -> uint32_t {
        return ptx::smem_addr(arr[(n / TPS) % NSS]) + ptx::sw128((n % TPS) * MB + t, chunk);
    };
    auto eta_at = [&](int n, int t) -> float { return s.eta[(n / TPS) % NSS][(n % TPS) * MB + t]; };

    // ---- state: W1^T rows hb + 16m + g (+8) x inputs 8pt + 2c (+1); W2 rows (same) x outputs
    const size_t init = p.init_per_batch ? (size_t)bh : (size_t)h;
    float w1[2][8][4], w2[2][8][4], b1r[2][2];
    {
        const float *W1 = p.W1 + init * D * DH;
        const float *W2 = p.W2 + init * DH * D;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int r0 = hb + 16 * m + g, r1 = r0 + 8;
#pragma unroll
            for (int pt = 0; pt < 8; ++pt) {
                const int i = 8 * pt + 2 * c;
                w1[m][pt][0] = W1[i * DH + r0];
                w1[m][pt][1] = W1[(i + 1) * DH + r0];
                w1[m][pt][2] = W1[i * DH + r1];
                w1[m][pt][3] = W1[(i + 1) * DH + r1];
                w2[m][pt][0] = W2[r0 * D + i];
                w2[m][pt][1] = W2[r0 * D + i + 1];
                w2[m][pt][2] = W2[r1 * D + i];
                w2[m][pt][3] = W2[r1 * D + i + 1];
            }
            b1r[m][0] = p.b1[init * DH + r0];
            b1r[m][1] = p.b1[init * DH + r1];
        }
    }
    float b2r[2] = {0.f, 0.f}, ga0 = 1.f, ga1 = 1.f, be0 = 0.f, be1 = 0.f, C1 = 0.f;
    // LayerNorm pivot: with the residual LayerNorm the scan runs on b2 - p, p = mean(b2) (LN and
    // its backward do not see a common shift of Z2), and p is added back to b2_final; the
    // one-pass sums of z and z^2 then stay free of cancellation when b2 has a large offset.
    float pivot = 0.f;
    if (lnw) {
        b2r[0] = p.b2[init * D + o0];
        b2r[1] = p.b2[init * D + o1];
        if (LN) {
            ga0 = p.gamma[(size_t)h * D + o0];
            ga1 = p.gamma[(size_t)h * D + o1];
            be0 = p.beta[(size_t)h * D + o0];
            be1 = p.beta[(size_t)h * D + o1];
            float part = ga0 * ga0 + ga1 * ga1, pb = b2r[0] + b2r[1];
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
                part += __shfl_xor_sync(0xffffffffu, part, o);
                pb += __shfl_xor_sync(0xffffffffu, pb, o);
            }
            if (lane == 0) {
                s.red[0][0][warp] = part;
                s.red[0][1][warp] = pb;
            }
            ptx::named_bar(kBarLn, 128);
            const float4 w4 = *reinterpret_cast<const float4 *>(s.red[0][0]);
            const float4 p4 = *reinterpret_cast<const float4 *>(s.red[0][1]);
            C1 = (w4.x + w4.y) + (w4.z + w4.w);
            pivot = ((p4.x + p4.y) + (p4.z + p4.w)) * (1.f / D);
            b2r[0] -= pivot;
            b2r[1] -= pivot;
            ptx::named_bar(kBarLn, 128);
        }
    }
    // inner-product loss -<f(k), v> (ai-feeds Modular TTT page): G2 = -V, or the LayerNorm
    // backward of the upstream -v; the same code path with the gamma^2, beta and k terms zeroed
    const float kf = p.ip ? 0.f : 1.f;
    C1 *= kf;
    const float g20 = kf * ga0 * ga0, g21 = kf * ga1 * ga1;
    const int tk = g >> 1, qh = g & 1;
    const int t_own = 8 * (tk >> 1) + 2 * c + (tk & 1);

    // C-fragment (rows = outputs o0/o1, cols = tokens) of a stage tile, transposed
    auto load_T = [&](float (*out)[4], const __nv_bfloat16 (*arr)[ST * D], int n) {
        uint32_t r[4];
        ptx::ldsm_x4_t(tile_addr(arr, n, (mat >> 1) * 8 + mrow, warp * 2 + (mat & 1)), r);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            out[u][0] = ptx::bf16_lo(r[2 * u]);
            out[u][1] = ptx::bf16_hi(r[2 * u]);
            out[u][2] = ptx::bf16_lo(r[2 * u + 1]);
            out[u][3] = ptx::bf16_hi(r[2 * u + 1]);
        }
    };
    // this warp's 32 hidden rows of W1^T X^T + b1 for the 16 tokens of a stage tile
    auto first_layer = [&](float (*acc)[2][4], const __nv_bfloat16 (*arr)[ST * D], int n) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                acc[m][u][0] = b1r[m][0]; acc[m][u][1] = b1r[m][0];
                acc[m][u][2] = b1r[m][1]; acc[m][u][3] = b1r[m][1];
            }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t r[4];   // B fragments (k = inputs 16q.., n = tokens): (t0, 2q), (t0, 2q+1), (t1, 2q), (t1, 2q+1)
            ptx::ldsm_x4(tile_addr(arr, n, (mat >> 1) * 8 + mrow, 2 * q + (mat & 1)), r);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const uint32_t a[4] = {ptx::pack_bf16(w1[m][2 * q][0], w1[m][2 * q][1]),
                                       ptx::pack_bf16(w1[m][2 * q][2], w1[m][2 * q][3]),
                                       ptx::pack_bf16(w1[m][2 * q + 1][0], w1[m][2 * q + 1][1]),
                                       ptx::pack_bf16(w1[m][2 * q + 1][2], w1[m][2 * q + 1][3])};
                ptx::mma_bf16(acc[m][0], a, r[0], r[1]);
                ptx::mma_bf16(acc[m][1], a, r[2], r[3]);
            }
        }
    };
    // rows = this warp's hidden units, cols = tokens  ->  bf16 [t][h] tile (transposed store)
    auto store_th = [&](uint32_t tile, const float (*x)[2][4]) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const uint32_t r[4] = {ptx::pack_bf16(x[m][0][0], x[m][0][1]), ptx::pack_bf16(x[m][0][2], x[m][0][3]),
                                   ptx::pack_bf16(x[m][1][0], x[m][1][1]), ptx::pack_bf16(x[m][1][2], x[m][1][3])};
            // matrices (h-block, t-block): (0,0), (1,0), (0,1), (1,1); stored rows = tokens
            ptx::stsm_x4_t(tile + xh_off((mat >> 1) * 8 + mrow, (hb + 16 * m) / 8 + (mat & 1)), r);
        }
    };
    // Zbar^T partial for the outputs of warp (warp & 3) = b + W2^T X^T over hidden units
    // 128 kh .. 128 kh + 127 (X from a [t][h] tile)
    auto second_layer = [&](float (*acc)[4], uint32_t xtile, float bo0, float bo1, int kh) {
        float hi[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            acc[u][0] = bo0; acc[u][1] = bo0; acc[u][2] = bo1; acc[u][3] = bo1;
            hi[u][0] = 0.f; hi[u][1] = 0.f; hi[u][2] = 0.f; hi[u][3] = 0.f;
        }
        const uint32_t wb = ptx::smem_addr(s.w2b);
#pragma unroll 4
        for (int q = 8 * kh; q < 8 * kh + 8; ++q) {
            uint32_t a[4], r[4];
            // A = W2^T (m = outputs, k = hidden 16q..): W2 is stored [h][o], so a transposed load of
            // matrices (o-block, h-block): (0,0), (1,0), (0,1), (1,1)
            ptx::ldsm_x4_t(wb + ptx::sw128(16 * q + 8 * (mat >> 1) + mrow, 2 * (warp & 3) + (mat & 1)), a);
            // B = X^T (k = hidden, n = tokens): (t0, chunk 2q), (t0, 2q+1), (t1, 2q), (t1, 2q+1)
            ptx::ldsm_x4(xtile + xh_off((mat >> 1) * 8 + mrow, 2 * q + (mat & 1)), r);
            float(*dst)[4] = (q & 1) ? hi : acc;
            ptx::mma_bf16(dst[0], a, r[0], r[1]);
            ptx::mma_bf16(dst[1], a, r[2], r[3]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[u][i] += hi[u][i];
    };
    // reduce-scatter of 8 per-token values over the 8 lanes sharing c
    auto rs8 = [&](const float *zs) -> float {
        float b4[4], b2v[2];
        {
            const bool hi = (lane >> 4) & 1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float snd = hi ? zs[i] : zs[4 + i];
                const float kp = hi ? zs[4 + i] : zs[i];
                b4[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 16);
            }
        }
        {
            const bool hi = (lane >> 3) & 1;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float snd = hi ? b4[i] : b4[2 + i];
                const float kp = hi ? b4[2 + i] : b4[i];
                b2v[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 8);
            }
        }
        const bool hi = (lane >> 2) & 1;
        const float snd = hi ? b2v[0] : b2v[1];
        const float kp = hi ? b2v[1] : b2v[0];
        return kp + __shfl_xor_sync(0xffffffffu, snd, 4);
    };

    const uint32_t x2t = ptx::smem_addr(s.x2), xb2t = ptx::smem_addr(s.xb2);

    wait_stage(0);
    for (int n = 0; n < N; ++n) {
        const int par = n & 1, st = n / TPS;
        if (n % TPS == 0 && n > 0) wait_stage(st);

        // ======== phase 1: first layer (key and query side), W2 copy, the Q K^T block
        float y1[2][2][4];
        float fq[2][2] = {{1.f, 1.f}, {1.f, 1.f}}, dn = 1.f;   // weight decay factors (below)
        uint32_t dz[2][2][2];   // GELU'(Z1) as bf16 pairs (it only scales G1, a bf16 operand)
        uint32_t xa[2][4];      // X2 = GELU(Z1) as bf16 A fragments (rows = hidden, k = tokens)
        {
        float z1[2][2][4];
        first_layer(z1, s.k, n);
        first_layer(y1, s.q, n);
        // weight decay (ai-feeds Modular TTT page; W1, W2 only, gradient at the mini-batch's
        // start): query token t reads f_t = 1 - lambda cum_t times W1, W2 (a prefix sum of eta
        // by a scan over the four lanes sharing g), and the carried weights are scaled by
        // dn = 1 - lambda sum eta before their updates
        if (WD) {
            const float a0 = eta_at(n, 2 * c), a1 = eta_at(n, 2 * c + 1);
            const float bb0 = eta_at(n, 2 * c + 8), bb1 = eta_at(n, 2 * c + 9);
            float ia = a0 + a1, ib = bb0 + bb1;
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                const float ta = __shfl_up_sync(0xffffffffu, ia, o, 4);
                const float tb = __shfl_up_sync(0xffffffffu, ib, o, 4);
                if (c >= o) {
                    ia += ta;
                    ib += tb;
                }
            }
            const float ta = __shfl_sync(0xffffffffu, ia, 3, 4);   // tokens 0..7
            const float tb = __shfl_sync(0xffffffffu, ib, 3, 4);   // tokens 8..15
            fq[0][0] = 1.f - p.wd * (ia - a1);
            fq[0][1] = 1.f - p.wd * ia;
            fq[1][0] = 1.f - p.wd * (ta + ib - bb1);
            fq[1][1] = 1.f - p.wd * (ta + ib);
            dn = 1.f - p.wd * (ta + tb);
            // Y1 = f (Q W1) + b1 from Y1 = Q W1 + b1
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float f = fq[u][i & 1];
                        y1[m][u][i] = fmaf(f, y1[m][u][i], (1.f - f) * b1r[m][i >> 1]);
                    }
        }
        // X2 also goes to the shared [t][h] tile
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            float y[2][4], dy[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) gelu_and_prime(z1[m][u][i], y[u][i], dy[u][i]);
            xa[m][0] = ptx::pack_bf16(y[0][0], y[0][1]);
            xa[m][1] = ptx::pack_bf16(y[0][2], y[0][3]);
            xa[m][2] = ptx::pack_bf16(y[1][0], y[1][1]);
            xa[m][3] = ptx::pack_bf16(y[1][2], y[1][3]);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                dz[m][u][0] = ptx::pack_bf16(dy[u][0], dy[u][1]);
                dz[m][u][1] = ptx::pack_bf16(dy[u][2], dy[u][3]);
            }
            // matrices (h-block, t-block): (0,0), (1,0), (0,1), (1,1); stored rows = tokens
            ptx::stsm_x4_t(x2t + xh_off((mat >> 1) * 8 + mrow, (hb + 16 * m) / 8 + (mat & 1)), xa[m]);
        }
        }
        {
            // W2 rows hb.. (bf16) into the [h][o] tile: matrices (h 0-7, o 16k..), (h 8-15, ..), (h 0-7, o 16k+8..), (h 8-15, ..)
            const uint32_t wb = ptx::smem_addr(s.w2b);
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t r[4] = {ptx::pack_bf16(w2[m][2 * k][0], w2[m][2 * k][1]),
                                           ptx::pack_bf16(w2[m][2 * k][2], w2[m][2 * k][3]),
                                           ptx::pack_bf16(w2[m][2 * k + 1][0], w2[m][2 * k + 1][1]),
                                           ptx::pack_bf16(w2[m][2 * k + 1][2], w2[m][2 * k + 1][3])};
                    ptx::stsm_x4(wb + ptx::sw128(hb + 16 * m + 8 * (mat & 1) + mrow, 2 * k + (mat >> 1)), r);
                }
        }
        if (warp == 4 || warp == 5) {
            // eta_s (Q_t . K_s + 1) [s <= t], source half (warp & 1)
            const int half = warp & 1;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t a[4], b[4];
                ptx::ldsm_x4(tile_addr(s.q, n, (mat & 1) * 8 + mrow, 2 * q + (mat >> 1)), a);
                ptx::ldsm_x4(tile_addr(s.k, n, half * 8 + mrow, 2 * q + (mat & 1)), b);
                ptx::mma_bf16(acc, a, b[0], b[1]);
            }
            const int s0 = half * 8 + 2 * c;
            const float e0 = eta_at(n, s0), e1 = eta_at(n, s0 + 1);
            const float v0 = s0 > g ? 0.f : e0 * (acc[0] + 1.f), v1 = s0 + 1 > g ? 0.f : e1 * (acc[1] + 1.f);
            const float v2 = s0 > g + 8 ? 0.f : e0 * (acc[2] + 1.f), v3 = s0 + 1 > g + 8 ? 0.f : e1 * (acc[3] + 1.f);
            *reinterpret_cast<uint2 *>(s.a1f[half][lane]) = make_uint2(ptx::pack_bf16(v0, v1), ptx::pack_bf16(v2, v3));
        }
        ptx::named_bar(kBarAll, kCompute * 32);

        // ======== phase 2: Z2 = X2 W2 + b2 (all warps, one hidden half each), then G2 (warps 0-3)
        float gm[2][4];      // G2^T for o0/o1 (warps 0-3)
        float vt[2][4];
        const float b2_start0 = b2r[0], b2_start1 = b2r[1];
        float z2[2][4];
        second_layer(z2, x2t, b2r[0], b2r[1], warp >> 2);   // b2r is zero on warps 4-7
        if (!lnw) {
            float4 *dst = reinterpret_cast<float4 *>(s.part2[warp & 3][lane]);
            dst[0] = make_float4(z2[0][0], z2[0][1], z2[0][2], z2[0][3]);
            dst[1] = make_float4(z2[1][0], z2[1][1], z2[1][2], z2[1][3]);
        }
        ptx::named_bar(kBarAll, kCompute * 32);
        if (lnw) {
            {
                const float4 p0 = reinterpret_cast<const float4 *>(s.part2[warp][lane])[0];
                const float4 p1 = reinterpret_cast<const float4 *>(s.part2[warp][lane])[1];
                z2[0][0] += p0.x; z2[0][1] += p0.y; z2[0][2] += p0.z; z2[0][3] += p0.w;
                z2[1][0] += p1.x; z2[1][1] += p1.y; z2[1][2] += p1.z; z2[1][3] += p1.w;
            }
            load_T(vt, s.v, n);
            if (LN) {
                float kt[2][4], gb[2][4];
                load_T(kt, s.k, n);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    gb[u][0] = ga0 * fmaf(kf, be0 + kt[u][0], -vt[u][0]);
                    gb[u][1] = ga0 * fmaf(kf, be0 + kt[u][1], -vt[u][1]);
                    gb[u][2] = ga1 * fmaf(kf, be1 + kt[u][2], -vt[u][2]);
                    gb[u][3] = ga1 * fmaf(kf, be1 + kt[u][3], -vt[u][3]);
                }
                float vs[24];
#pragma unroll
                for (int t4 = 0; t4 < 4; ++t4) {
                    const int u = t4 >> 1, e = t4 & 1;
                    const float a0z = z2[u][e], a1z = z2[u][2 + e];
                    const float a0 = g20 * a0z, a1 = g21 * a1z;
                    vs[t4 * 6 + 0] = a0z + a1z;
                    vs[t4 * 6 + 1] = fmaf(a0z, a0z, a1z * a1z);
                    vs[t4 * 6 + 2] = a0 + a1;
                    vs[t4 * 6 + 3] = fmaf(a0, a0z, a1 * a1z);
                    vs[t4 * 6 + 4] = fmaf(gb[u][e], a0z, gb[u][2 + e] * a1z);
                    vs[t4 * 6 + 5] = gb[u][e] + gb[u][2 + e];
                }
                float a12[12], a6[6], a3[3];
                {
                    const bool hi = (lane >> 4) & 1;
#pragma unroll
                    for (int i = 0; i < 12; ++i) {
                        const float snd = hi ? vs[i] : vs[12 + i];
                        const float kp = hi ? vs[12 + i] : vs[i];
                        a12[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 16);
                    }
                }
                {
                    const bool hi = (lane >> 3) & 1;
#pragma unroll
                    for (int i = 0; i < 6; ++i) {
                        const float snd = hi ? a12[i] : a12[6 + i];
                        const float kp = hi ? a12[6 + i] : a12[i];
                        a6[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 8);
                    }
                }
                {
                    const bool hi = (lane >> 2) & 1;
#pragma unroll
                    for (int i = 0; i < 3; ++i) {
                        const float snd = hi ? a6[i] : a6[3 + i];
                        const float kp = hi ? a6[3 + i] : a6[i];
                        a3[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 4);
                    }
                }
#pragma unroll
                for (int i = 0; i < 3; ++i) s.red[par][t_own][4 * (3 * qh + i) + warp] = a3[i];
                ptx::named_bar(kBarLn, 128);
                float tot[3];
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const float4 w4 = *reinterpret_cast<const float4 *>(&s.red[par][t_own][4 * (3 * qh + i)]);
                    tot[i] = (w4.x + w4.y) + (w4.z + w4.w);
                }
                float S[6];
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const float o = __shfl_xor_sync(0xffffffffu, tot[i], 4);
                    S[i] = qh ? o : tot[i];
                    S[3 + i] = qh ? tot[i] : o;
                }
                const float mu = S[0] * (1.f / D);
                const float var = fmaxf(S[1] * (1.f / D) - mu * mu, 0.f);
                const float r = rsqrtf(var + p.eps);
                const float sg2zc = S[2] - mu * C1;
                const float sg2zc2 = S[3] - 2.f * mu * S[2] + mu * mu * C1;
                const float sgbzc = S[4] - mu * S[5];
                const float m1 = (r * sg2zc + S[5]) * (1.f / D);
                const float m2 = (r * r * sg2zc2 + r * sgbzc) * (1.f / D);
                const float co_a = r * r, co_b = r * r * m2, co_e = r * m1;
#pragma unroll
                for (int tq = 0; tq < 4; ++tq) {
                    const int src = c + 8 * tq;
                    const float mu_t = __shfl_sync(0xffffffffu, mu, src);
                    const float a_t = __shfl_sync(0xffffffffu, co_a, src);
                    const float b_t = __shfl_sync(0xffffffffu, co_b, src);
                    const float r_t = __shfl_sync(0xffffffffu, r, src);
                    const float e_t = __shfl_sync(0xffffffffu, co_e, src);
                    const int u = tq >> 1, e = tq & 1;
                    const float zc0 = z2[u][e] - mu_t, zc1 = z2[u][2 + e] - mu_t;
                    gm[u][e] = fmaf(zc0, fmaf(a_t, g20, -b_t), fmaf(r_t, gb[u][e], -e_t));
                    gm[u][2 + e] = fmaf(zc1, fmaf(a_t, g21, -b_t), fmaf(r_t, gb[u][2 + e], -e_t));
                }
            } else {
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) gm[u][i] = fmaf(z2[u][i], kf, -vt[u][i]);
            }
            // publish G2 and -eta G2 as [t][o] tiles; b2 -= eta^T G2
            const int s0 = 2 * c;
            const float e00 = eta_at(n, s0), e01 = eta_at(n, s0 + 1);
            const float e10 = eta_at(n, s0 + 8), e11 = eta_at(n, s0 + 9);
            const uint32_t r[4] = {ptx::pack_bf16(gm[0][0], gm[0][1]), ptx::pack_bf16(gm[0][2], gm[0][3]),
                                   ptx::pack_bf16(gm[1][0], gm[1][1]), ptx::pack_bf16(gm[1][2], gm[1][3])};
            const uint32_t re[4] = {ptx::pack_bf16(-e00 * gm[0][0], -e01 * gm[0][1]),
                                    ptx::pack_bf16(-e00 * gm[0][2], -e01 * gm[0][3]),
                                    ptx::pack_bf16(-e10 * gm[1][0], -e11 * gm[1][1]),
                                    ptx::pack_bf16(-e10 * gm[1][2], -e11 * gm[1][3])};
            const uint32_t off = ptx::sw128((mat >> 1) * 8 + mrow, warp * 2 + (mat & 1));
            ptx::stsm_x4_t(ptx::smem_addr(s.g2) + off, r);
            ptx::stsm_x4_t(ptx::smem_addr(s.eg2) + off, re);
            float d0 = e00 * gm[0][0] + e01 * gm[0][1] + e10 * gm[1][0] + e11 * gm[1][1];
            float d1 = e00 * gm[0][2] + e01 * gm[0][3] + e10 * gm[1][2] + e11 * gm[1][3];
            d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
            d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
            b2r[0] -= d0;
            b2r[1] -= d1;
        }
        ptx::named_bar(kBarAll, kCompute * 32);

        // ======== phase 3 (all): G1, first output layer, both state updates
        float g1[2][2][4];
        {
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) g1[m][u][i] = 0.f;
            const uint32_t gt = ptx::smem_addr(s.g2);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t r[4];   // B = G2^T (k = outputs 16k.., n = tokens): (t0, 2k), (t0, 2k+1), (t1, 2k), (t1, 2k+1)
                ptx::ldsm_x4(gt + ptx::sw128((mat >> 1) * 8 + mrow, 2 * k + (mat & 1)), r);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const uint32_t a[4] = {ptx::pack_bf16(w2[m][2 * k][0], w2[m][2 * k][1]),
                                           ptx::pack_bf16(w2[m][2 * k][2], w2[m][2 * k][3]),
                                           ptx::pack_bf16(w2[m][2 * k + 1][0], w2[m][2 * k + 1][1]),
                                           ptx::pack_bf16(w2[m][2 * k + 1][2], w2[m][2 * k + 1][3])};
                    ptx::mma_bf16(g1[m][0], a, r[0], r[1]);
                    ptx::mma_bf16(g1[m][1], a, r[2], r[3]);
                }
            }
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        g1[m][u][i] *= (i & 1) ? ptx::bf16_hi(dz[m][u][i >> 1]) : ptx::bf16_lo(dz[m][u][i >> 1]);
        }
        // first output layer: Zb1^T = Y1^T - G1^T (eta (Q K^T + 1) mask)^T, Xb2 = GELU(Zb1)
        {
            const uint2 f0 = *reinterpret_cast<const uint2 *>(s.a1f[0][lane]);
            const uint2 f1 = *reinterpret_cast<const uint2 *>(s.a1f[1][lane]);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const uint32_t a[4] = {ptx::pack_bf16(-g1[m][0][0], -g1[m][0][1]),
                                       ptx::pack_bf16(-g1[m][0][2], -g1[m][0][3]),
                                       ptx::pack_bf16(-g1[m][1][0], -g1[m][1][1]),
                                       ptx::pack_bf16(-g1[m][1][2], -g1[m][1][3])};
                ptx::mma_bf16(y1[m][0], a, f0.x, f1.x);
                ptx::mma_bf16(y1[m][1], a, f0.y, f1.y);
            }
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) y1[m][u][i] = gelu(y1[m][u][i]);
            store_th(xb2t, y1);
        }
        // W1^T += (-eta G1)^T K,  b1 -= eta^T G1   (W1 scaled by dn first with weight decay)
        {
            if (WD)
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
#pragma unroll
                        for (int i = 0; i < 4; ++i) w1[m][q][i] *= dn;
            const int s0 = 2 * c;
            const float e00 = eta_at(n, s0), e01 = eta_at(n, s0 + 1);
            const float e10 = eta_at(n, s0 + 8), e11 = eta_at(n, s0 + 9);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const uint32_t a[4] = {ptx::pack_bf16(-e00 * g1[m][0][0], -e01 * g1[m][0][1]),
                                       ptx::pack_bf16(-e00 * g1[m][0][2], -e01 * g1[m][0][3]),
                                       ptx::pack_bf16(-e10 * g1[m][1][0], -e11 * g1[m][1][1]),
                                       ptx::pack_bf16(-e10 * g1[m][1][2], -e11 * g1[m][1][3])};
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    uint32_t r[4];   // B = K (k = tokens, n = inputs): (s0-7, 2pp), (s8-15, 2pp), (s0-7, 2pp+1), (s8-15, 2pp+1)
                    ptx::ldsm_x4_t(tile_addr(s.k, n, (mat & 1) * 8 + mrow, 2 * pp + (mat >> 1)), r);
                    ptx::mma_bf16(w1[m][2 * pp], a, r[0], r[1]);
                    ptx::mma_bf16(w1[m][2 * pp + 1], a, r[2], r[3]);
                }
                float d0 = e00 * g1[m][0][0] + e01 * g1[m][0][1] + e10 * g1[m][1][0] + e11 * g1[m][1][1];
                float d1 = e00 * g1[m][0][2] + e01 * g1[m][0][3] + e10 * g1[m][1][2] + e11 * g1[m][1][3];
                d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
                d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
                d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
                d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
                b1r[m][0] -= d0;
                b1r[m][1] -= d1;
            }
        }
        // W2 += X2^T (-eta G2)   (A = X2^T rows = hidden, k = tokens; B = -eta G2 [t][o]); W2 is
        // no longer read as the step's starting weights (G1 above used it): scale by dn first
        {
            if (WD)
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
#pragma unroll
                        for (int i = 0; i < 4; ++i) w2[m][q][i] *= dn;
            const uint32_t eg = ptx::smem_addr(s.eg2);
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                uint32_t r[4];   // (t0-7, o-chunk 2pp), (t8-15, 2pp), (t0-7, 2pp+1), (t8-15, 2pp+1)
                ptx::ldsm_x4_t(eg + ptx::sw128((mat & 1) * 8 + mrow, 2 * pp + (mat >> 1)), r);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    ptx::mma_bf16(w2[m][2 * pp], xa[m], r[0], r[1]);
                    ptx::mma_bf16(w2[m][2 * pp + 1], xa[m], r[2], r[3]);
                }
            }
        }
        ptx::named_bar(kBarAll, kCompute * 32);

        // ======== phase 4: second output layer (all warps, one hidden half each), its 16 x 16
        // block eta_s (Xb2_t . X2_s + 1) [s <= t] (partials on warps 4-7), then warps 0-3 finish
        float zb[2][4];
        second_layer(zb, xb2t, b2_start0, b2_start1, warp >> 2);
        if (!lnw) {
            const int half = warp & 1, kq = (warp >> 1) & 1;   // source half, hidden half
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, ac2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int q = 8 * kq; q < 8 * kq + 8; ++q) {
                uint32_t a[4], b[4];
                // A = Xb2 rows t, k = hidden: (t0, 2q), (t1, 2q), (t0, 2q+1), (t1, 2q+1)
                ptx::ldsm_x4(xb2t + xh_off((mat & 1) * 8 + mrow, 2 * q + (mat >> 1)), a);
                // B = X2 rows s (this half), k = hidden: (s, 2q), (s, 2q+1)
                ptx::ldsm_x4(x2t + xh_off(half * 8 + mrow, 2 * q + (mat & 1)), b);
                ptx::mma_bf16((q & 1) ? ac2 : acc, a, b[0], b[1]);
            }
            *reinterpret_cast<float4 *>(s.parta2[half][kq][lane]) =
                make_float4(acc[0] + ac2[0], acc[1] + ac2[1], acc[2] + ac2[2], acc[3] + ac2[3]);
            float4 *dst = reinterpret_cast<float4 *>(s.part2[warp & 3][lane]);
            dst[0] = make_float4(zb[0][0], zb[0][1], zb[0][2], zb[0][3]);
            dst[1] = make_float4(zb[1][0], zb[1][1], zb[1][2], zb[1][3]);
        }
        ptx::named_bar(kBarAll, kCompute * 32);
        if (lnw) {
            {
                const float4 p0 = reinterpret_cast<const float4 *>(s.part2[warp][lane])[0];
                const float4 p1 = reinterpret_cast<const float4 *>(s.part2[warp][lane])[1];
                zb[0][0] += p0.x; zb[0][1] += p0.y; zb[0][2] += p0.z; zb[0][3] += p0.w;
                zb[1][0] += p1.x; zb[1][1] += p1.y; zb[1][2] += p1.z; zb[1][3] += p1.w;
            }
            if (WD)   // Zb2 = f (Xb2 W2) + b2 from Xb2 W2 + b2 (the starting b2)
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float f = fq[u][i & 1];
                        zb[u][i] = fmaf(f, zb[u][i], (1.f - f) * (i < 2 ? b2_start0 : b2_start1));
                    }
            // B fragments (k = source s, n = target t) of the block, per source half
            uint32_t f[2][2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const float4 p = *reinterpret_cast<const float4 *>(s.parta2[half][0][lane]);
                const float4 q2 = *reinterpret_cast<const float4 *>(s.parta2[half][1][lane]);
                const int s0 = half * 8 + 2 * c;
                const float e0 = eta_at(n, s0), e1 = eta_at(n, s0 + 1);
                const float v0 = s0 > g ? 0.f : e0 * (p.x + q2.x + 1.f);
                const float v1 = s0 + 1 > g ? 0.f : e1 * (p.y + q2.y + 1.f);
                const float v2 = s0 > g + 8 ? 0.f : e0 * (p.z + q2.z + 1.f);
                const float v3 = s0 + 1 > g + 8 ? 0.f : e1 * (p.w + q2.w + 1.f);
                f[half][0] = ptx::pack_bf16(v0, v1);
                f[half][1] = ptx::pack_bf16(v2, v3);
            }
            const uint32_t a[4] = {ptx::pack_bf16(-gm[0][0], -gm[0][1]), ptx::pack_bf16(-gm[0][2], -gm[0][3]),
                                   ptx::pack_bf16(-gm[1][0], -gm[1][1]), ptx::pack_bf16(-gm[1][2], -gm[1][3])};
            ptx::mma_bf16(zb[0], a, f[0][0], f[1][0]);
            ptx::mma_bf16(zb[1], a, f[0][1], f[1][1]);
            float z[2][4];
            if (LN) {
                float zs[8];
#pragma unroll
                for (int tq = 0; tq < 4; ++tq) {
                    const int u = tq >> 1, e = tq & 1;
                    const float z0 = zb[u][e], z1v = zb[u][2 + e];
                    zs[tq * 2 + 0] = z0 + z1v;
                    zs[tq * 2 + 1] = fmaf(z0, z0, z1v * z1v);
                }
                s.zred[par][t_own][4 * qh + warp] = rs8(zs);
                ptx::named_bar(kBarLn, 128);
                const float4 w4 = *reinterpret_cast<const float4 *>(&s.zred[par][t_own][4 * qh]);
                const float tot = (w4.x + w4.y) + (w4.z + w4.w);
                const float oth = __shfl_xor_sync(0xffffffffu, tot, 4);
                const float s1 = qh ? oth : tot, s2 = qh ? tot : oth;
                const float mu = s1 * (1.f / D);
                const float var = fmaxf(s2 * (1.f / D) - mu * mu, 0.f);
                const float r = rsqrtf(var + p.eps);
                float qt[2][4];
                load_T(qt, s.q, n);
#pragma unroll
                for (int tq = 0; tq < 4; ++tq) {
                    const float m_t = __shfl_sync(0xffffffffu, mu, c + 8 * tq);
                    const float r_t = __shfl_sync(0xffffffffu, r, c + 8 * tq);
                    const int u = tq >> 1, e = tq & 1;
                    z[u][e] = qt[u][e] + fmaf(ga0 * (zb[u][e] - m_t), r_t, be0);
                    z[u][2 + e] = qt[u][2 + e] + fmaf(ga1 * (zb[u][2 + e] - m_t), r_t, be1);
                }
            } else {
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) z[u][i] = zb[u][i];
            }
            const uint32_t r[4] = {ptx::pack_bf16(z[0][0], z[0][1]), ptx::pack_bf16(z[0][2], z[0][3]),
                                   ptx::pack_bf16(z[1][0], z[1][1]), ptx::pack_bf16(z[1][2], z[1][3])};
            const uint32_t zt = ptx::smem_addr(s.zst);
            ptx::stsm_x4_t(zt + ptx::sw128((mat >> 1) * 8 + mrow, warp * 2 + (mat & 1)), r);
            ptx::named_bar(kBarLn, 128);
            // 16 rows x 128 bytes, one 16-byte chunk per thread of warps 0-3
            {
                const int row = tid >> 3, ch = tid & 7;
                uint4 val;
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                             : "r"(zt + ptx::sw128(row, ch)));
                uint4 *dst = reinterpret_cast<uint4 *>(Zg + ((size_t)bh * p.L + (size_t)n * MB + row) * D) + ch;
                *dst = val;
            }
            // warps 4-7 have not read stage st since the barrier before this step's output
            // layer, warps 0-3 since the barrier above: refill its slot
            if (tid == 0 && n % TPS == TPS - 1 && st + NSS < nissue && !aborted) {
                ptx::fence_proxy_async();
                issue_stage(st + NSS);
                issued = st + NSS + 1;
            }
        }
    }
    // copies still in flight (only after a wait ran out) must land before the CTA exits
    if (tid == 0)
        for (int st = max(0, issued - NSS); st < issued; ++st)
            ptx::mbar_wait_bounded(ptx::smem_addr(&s.full[st % NSS]), (st / NSS) & 1, kDrainNs);

    // ---- final state
    float *W1f = p.W1f + (size_t)bh * D * DH;
    float *W2f = p.W2f + (size_t)bh * DH * D;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int r0 = hb + 16 * m + g, r1 = r0 + 8;
#pragma unroll
        for (int pt = 0; pt < 8; ++pt) {
            const int i = 8 * pt + 2 * c;
            W1f[i * DH + r0] = w1[m][pt][0];
            W1f[(i + 1) * DH + r0] = w1[m][pt][1];
            W1f[i * DH + r1] = w1[m][pt][2];
            W1f[(i + 1) * DH + r1] = w1[m][pt][3];
            W2f[r0 * D + i] = w2[m][pt][0];
            W2f[r0 * D + i + 1] = w2[m][pt][1];
            W2f[r1 * D + i] = w2[m][pt][2];
            W2f[r1 * D + i + 1] = w2[m][pt][3];
        }
        if (c == 0) {
            p.b1f[(size_t)bh * DH + r0] = b1r[m][0];
            p.b1f[(size_t)bh * DH + r1] = b1r[m][1];
        }
    }
    if (lnw && c == 0) {
        p.b2f[(size_t)bh * D + o0] = b2r[0] + pivot;
        p.b2f[(size_t)bh * D + o1] = b2r[1] + pivot;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_mlp()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [BH][L][64] bf16 viewed as a 3-D tensor; boxes of 64 tokens, 128-byte swizzle.
bool make_map_mlp(CUtensorMap *m, const void *base, int L, int BH)
{
    auto enc = get_encode_mlp();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)ST, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool mlp_tc_supported(const ttt_desc &d)
{
    return d.io_dtype == TTT_BF16 && d.d == D && d.d_hidden == DH && d.mini_batch == MB;
}

cudaError_t launch_mlp_tc(const MlpArgs &a)
{
    const ttt_desc &d = a.desc;
    const int BH = call_rows(d);
    CUtensorMap mq, mk, mv;
    if (!make_map_mlp(&mq, a.Q, d.L, BH) || !make_map_mlp(&mk, a.K, d.L, BH) || !make_map_mlp(&mv, a.V, d.L, BH))
        return cudaErrorInvalidValue;
    Params p;
    p.H = d.H;
    p.L = d.L;
    p.N = d.L / MB;
    p.NST = (d.L + ST - 1) / ST;
    p.init_per_batch = d.init_per_batch;
    p.eps = d.ln_eps;
    p.wait_ns = wait_timeout_ns();
    p.withhold_loads = withhold_loads();
    p.eta = a.eta;
    p.W1 = a.W1_0;
    p.b1 = a.b1_0;
    p.W2 = a.W2_0;
    p.b2 = a.b2_0;
    p.gamma = a.gamma;
    p.beta = a.beta;
    p.W1f = a.W1_f;
    p.b1f = a.b1_f;
    p.W2f = a.W2_f;
    p.b2f = a.b2_f;
    p.status = a.status;
    p.hoff = head_offset(d);
    p.ip = d.loss == TTT_LOSS_INNER_PRODUCT;
    p.wd = d.weight_decay;
    const size_t smem = sizeof(Smem) + 1024;
    const bool wd = d.weight_decay != 0.f;
    auto kern = d.residual_ln ? (wd ? mlp_fused_kernel<true, true> : mlp_fused_kernel<true, false>)
                              : (wd ? mlp_fused_kernel<false, true> : mlp_fused_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<BH, kThreads, smem, a.stream>>>(mq, mk, mv, p, static_cast<__nv_bfloat16 *>(a.Z));
    return cudaGetLastError();
}

}  // namespace ttt
