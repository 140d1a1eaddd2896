// ttt_linear_tc.cu -- fused TTT-Linear forward for bf16 I/O, d = 64, b = 16.
//
// The method (damodev.csdn.net TTT article, sections 3.1 and 4.1-4.2; residual
// LayerNorm of the lryc.cn TTT article, section 2.1): per (batch, head) the
// fast weights (W, c) are updated once per mini-batch of 16 tokens, every
// token's gradient taken at the mini-batch's starting weights, and each
// output read with the weights after its own token's update.  With
//   P_n = K_n W_n + 1 c_n                        (key-side forward, 16 x 64)
//   G_n = P_n - V_n  or  LNbwd(P_n; V_n - K_n)   (per-token gradient)
//   W_{n+1} = W_n - K_n^T diag(eta_n) G_n,  c_{n+1} = c_n - eta_n^T G_n
//   Z_n = f_out(Q_n W_n + 1 c_n - (tril(Q_n K_n^T + 1) diag(eta_n)) G_n)
// the only sequential dependency is P_n -> G_n -> W_{n+1} -> P_{n+1}.
//
// B300 design.  One CTA per (batch, head); five warps:
//   * warp 4 streams 64-token stages of Q, K, V (TMA, 128-byte swizzle) and
//     eta (bulk copy) into a 6-deep shared-memory ring, mbarrier-synchronised;
//   * warps 0-3 each own 16 output features of the state.  W^T lives in
//     registers as fp32 mma accumulators for the whole scan; every contraction
//     is a warp-level bf16 MMA on register fragments, so the recurrence never
//     leaves the register file.  The key-side product of the NEXT mini-batch
//     is taken one step early, from W_n:
//         P_{n+1} = (K_{n+1} W_n + c_n) - ((K_{n+1} K_n^T + 1) diag(eta_n)) G_n,
//     which is exact, so the critical chain per mini-batch is only
//     G_n -> a 16x16x16 correction -> G_{n+1}; the d x d update and both d x d
//     products overlap it.
//   * the input-only 16x16 blocks Q_n K_n^T and K_{n+1} K_n^T are computed one
//     mini-batch ahead, split over the four math warps, and exchanged through
//     shared memory as ready-made MMA operand fragments;
//   * LayerNorm statistics are reduced with a warp reduce-scatter plus one
//     shared-memory exchange; the backward statistics use a single pass
//     (sums of z, z^2, g^2 z, g^2 z^2, g b' z, g b' with b' = beta - v + k).
//   * Z tiles are transposed back with stmatrix into a swizzled staging ring
//     and written by TMA stores.
// Every mbarrier wait is bounded; a wait that runs out sets the library's
// failure flag and the kernel finishes without waiting again.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int D = 64;           // head dim
constexpr int MB = 16;          // mini-batch
constexpr int ST = 64;          // tokens per pipeline stage
constexpr int TPS = ST / MB;    // mini-batches per stage
constexpr int NSS = 6;          // stages in the ring
constexpr int NZ = 4;           // Z staging tiles
constexpr int kMathThreads = 128;
constexpr int kThreads = 160;
constexpr uint32_t kStageTileBytes = ST * D * 2;   // 8 KB

struct __align__(1024) Smem {
    __nv_bfloat16 q[NSS][ST * D];
    __nv_bfloat16 k[NSS][ST * D];
    __nv_bfloat16 v[NSS][ST * D];
    __nv_bfloat16 z[NZ][MB * D];
    float eta[NSS][ST];
    uint32_t sfrag[3][2][2][32][2];   // [step % 3][0: chain, 1: output][s half][lane][t n-tile]
    float red[2][MB][8][4];           // [parity][token][quantity][warp]
    float zred[2][MB][2][4];          // [parity][token][sum z, sum z^2][warp]
    unsigned long long full[NSS];
    unsigned long long empty[NSS];
    int abort_flag;
};

struct Params {
    int H, L, ln;
    float eps;
    long long wait_ns;       // bound of every mbarrier wait
    int withhold_loads;      // test hook: the producer issues no copies
    const float *eta, *W0, *b0, *gamma, *beta;
    float *Wf, *bf;
    unsigned int *status;
    int init_per_batch;
};

// Bound of the final wait for copies still in flight (they land in microseconds).
constexpr long long kDrainNs = 1000000000ll;
constexpr long long kDefaultWaitNs = 1000000000ll;

template <bool LN>
__global__ void __launch_bounds__(kThreads, 1)
linear_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmZ,
                    Params p)
{
    extern __shared__ unsigned char smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, h = bh % p.H;
    const int N = p.L / MB;                 // mini-batches
    const int NST = (p.L + ST - 1) / ST;    // stages

    if (tid == 0) {
        for (int i = 0; i < NSS; ++i) {
            ptx::mbar_init(ptx::smem_addr(&s.full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&s.empty[i]), 1);
        }
        s.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------------ producer
    if (warp == 4) {
        if (lane == 0) {
            ptx::prefetch_tmap(&tmQ);
            ptx::prefetch_tmap(&tmK);
            ptx::prefetch_tmap(&tmV);
            const float *eta_bh = p.eta + (size_t)bh * p.L;
            int issued = 0;
            for (int st = 0; st < (p.withhold_loads ? 0 : NST); ++st) {
                const int b = st % NSS;
                if (st >= NSS) {
                    if (*(volatile int *)&s.abort_flag) break;
                    if (!ptx::mbar_wait_bounded(ptx::smem_addr(&s.empty[b]), ((st / NSS) - 1) & 1,
                                                p.wait_ns)) {
                        *(volatile int *)&s.abort_flag = 1;
                        atomicOr(p.status, kStatusTimeout);
                        break;
                    }
                }
                const int ntok = min(ST, p.L - st * ST);
                const uint32_t fb = ptx::smem_addr(&s.full[b]);
                ptx::mbar_arrive_expect_tx(fb, 3 * kStageTileBytes + ntok * 4);
                ptx::tma_load_3d(ptx::smem_addr(s.q[b]), &tmQ, fb, 0, st * ST, bh);
                ptx::tma_load_3d(ptx::smem_addr(s.k[b]), &tmK, fb, 0, st * ST, bh);
                ptx::tma_load_3d(ptx::smem_addr(s.v[b]), &tmV, fb, 0, st * ST, bh);
                ptx::bulk_load(ptx::smem_addr(s.eta[b]), eta_bh + st * ST, ntok * 4, fb);
                issued = st + 1;
            }
            // every copy issued must land before the CTA may exit
            for (int st = max(0, issued - NSS); st < issued; ++st)
                ptx::mbar_wait_bounded(ptx::smem_addr(&s.full[st % NSS]), (st / NSS) & 1, kDrainNs);
        }
        return;
    }

    // ------------------------------------------------------------------ math warps
    const int g = lane >> 2, c = lane & 3;
    const int j0 = warp * 16 + g, j1 = j0 + 8;      // this thread's two features
    const long long lim = p.wait_ns;
    bool aborted = false;

    auto wait_stage = [&](int st) {
        if (aborted) return;
        if (*(volatile int *)&s.abort_flag) { aborted = true; return; }
        if (!ptx::mbar_wait_bounded(ptx::smem_addr(&s.full[st % NSS]), (st / NSS) & 1, lim)) {
            aborted = true;
            *(volatile int *)&s.abort_flag = 1;
            atomicOr(p.status, kStatusTimeout);
        }
    };
    // shared-memory byte address of row `t` (mini-batch n) / 16-byte chunk of a tile
    auto tile_addr = [&](const __nv_bfloat16 (*arr)[ST * D], int n, int t, int chunk) -> uint32_t {
        const int st = n / TPS;
        return ptx::smem_addr(arr[st % NSS]) + ptx::sw128((n % TPS) * MB + t, chunk);
    };
    auto eta_at = [&](int n, int t) -> float { return s.eta[(n / TPS) % NSS][(n % TPS) * MB + t]; };

    // ---- initial state: W^T rows j0/j1 as fp32 accumulators, c, LN params
    float wt[8][4];
    {
        const size_t init = p.init_per_batch ? (size_t)bh : (size_t)h;
        const float *W0 = p.W0 + init * D * D;
#pragma unroll
        for (int pt = 0; pt < 8; ++pt) {
            const int i = pt * 8 + 2 * c;
            wt[pt][0] = W0[i * D + j0];
            wt[pt][1] = W0[(i + 1) * D + j0];
            wt[pt][2] = W0[i * D + j1];
            wt[pt][3] = W0[(i + 1) * D + j1];
        }
    }
    float cb0 = p.b0[(p.init_per_batch ? (size_t)bh : (size_t)h) * D + j0];
    float cb1 = p.b0[(p.init_per_batch ? (size_t)bh : (size_t)h) * D + j1];
    float ga0 = 1.f, ga1 = 1.f, be0 = 0.f, be1 = 0.f, C1 = 0.f;
    if (LN) {
        ga0 = p.gamma[(size_t)h * D + j0];
        ga1 = p.gamma[(size_t)h * D + j1];
        be0 = p.beta[(size_t)h * D + j0];
        be1 = p.beta[(size_t)h * D + j1];
        for (int j = 0; j < D; ++j) {
            const float gj = p.gamma[(size_t)h * D + j];
            C1 = fmaf(gj, gj, C1);
        }
    }
    uint32_t wa[4][4];   // bf16 A fragments of W^T, k-steps of 16 input features
    auto pack_w = [&]() {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            wa[q][0] = ptx::pack_bf16(wt[2 * q][0], wt[2 * q][1]);
            wa[q][1] = ptx::pack_bf16(wt[2 * q][2], wt[2 * q][3]);
            wa[q][2] = ptx::pack_bf16(wt[2 * q + 1][0], wt[2 * q + 1][1]);
            wa[q][3] = ptx::pack_bf16(wt[2 * q + 1][2], wt[2 * q + 1][3]);
        }
    };
    pack_w();

    // acc[u][*] = W^T X_n^T (+ c) for a 16-token tile X of mini-batch n
    auto product = [&](float (*acc)[4], const __nv_bfloat16 (*arr)[ST * D], int n) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            acc[u][0] = cb0; acc[u][1] = cb0; acc[u][2] = cb1; acc[u][3] = cb1;
        }
        const int mrow = lane & 7, mat = lane >> 3;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // matrices: (t-block 0, i-chunk 2q), (t0, 2q+1), (t1, 2q), (t1, 2q+1)
            uint32_t r[4];
            ptx::ldsm_x4(tile_addr(arr, n, (mat >> 1) * 8 + mrow, 2 * q + (mat & 1)), r);
            ptx::mma_bf16(acc[0], wa[q], r[0], r[1]);
            ptx::mma_bf16(acc[1], wa[q], r[2], r[3]);
        }
    };

    // C-fragment layout (rows = features j0/j1, cols = tokens) of a bf16 tile, transposed
    auto load_T = [&](float (*out)[4], const __nv_bfloat16 (*arr)[ST * D], int n) {
        const int mrow = lane & 7, mat = lane >> 3;
        // matrices: (t-block 0, j-block 0), (t0, j1), (t1, j0), (t1, j1)
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

    // Input-only 16x16 blocks for mini-batch n, as B fragments (k = source
    // token s, n = target token t):
    //   chain : eta_s (K_{n+1}[t] . K_n[s] + 1)
    //   output: eta_s (Q_n[t] . K_n[s] + 1) [s <= t]
    // warp w: matrix (w >> 1) (0 output, 1 chain), source half (w & 1).
    auto compute_sfrag = [&](int n, int par) {
        const int which = warp >> 1, half = warp & 1;   // which: 0 output, 1 chain
        if (which == 1 && n + 1 >= N) return;
        const __nv_bfloat16(*A)[ST * D] = which ? s.k : s.q;
        const int na = which ? n + 1 : n;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int mrow = lane & 7, mat = lane >> 3;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // A = rows t of the target tile, k = features 16q..16q+15
            uint32_t a[4];
            // matrices: (t0, chunk 2q), (t1, 2q), (t0, 2q+1), (t1, 2q+1)
            ptx::ldsm_x4(tile_addr(A, na, (mat & 1) * 8 + mrow, 2 * q + (mat >> 1)), a);
            // B = K_n rows s in [8*half, 8*half+8), k = features: (s, chunk 2q), (s, 2q+1)
            uint32_t b[4];
            ptx::ldsm_x4(tile_addr(s.k, n, half * 8 + mrow, 2 * q + (mat & 1)), b);
            ptx::mma_bf16(acc, a, b[0], b[1]);
        }
        // acc: rows t = g (acc0,1), g + 8 (acc2,3); cols s = 8 half + 2c, +1
        const int s0 = half * 8 + 2 * c;
        const float e0 = eta_at(n, s0), e1 = eta_at(n, s0 + 1);
        float v[4];
        v[0] = e0 * (acc[0] + 1.f);
        v[1] = e1 * (acc[1] + 1.f);
        v[2] = e0 * (acc[2] + 1.f);
        v[3] = e1 * (acc[3] + 1.f);
        if (which == 0) {   // causal mask s <= t
            if (s0 > g) v[0] = 0.f;
            if (s0 + 1 > g) v[1] = 0.f;
            if (s0 > g + 8) v[2] = 0.f;
            if (s0 + 1 > g + 8) v[3] = 0.f;
        }
        uint32_t *dst = s.sfrag[par][which ? 0 : 1][half][lane];
        dst[0] = ptx::pack_bf16(v[0], v[1]);   // t n-tile 0
        dst[1] = ptx::pack_bf16(v[2], v[3]);   // t n-tile 1
    };
    auto read_sfrag = [&](int par, int which, uint32_t (*b)[2]) {   // b[u][half]
        const uint32_t *f0 = s.sfrag[par][which][0][lane];
        const uint32_t *f1 = s.sfrag[par][which][1][lane];
        b[0][0] = f0[0]; b[1][0] = f0[1];
        b[0][1] = f1[0]; b[1][1] = f1[1];
    };

    // ---- prologue: P_0, block fragments of mini-batch 0
    wait_stage(0);
    float pacc[2][4];
    product(pacc, s.k, 0);
    compute_sfrag(0, 0);
    ptx::named_bar(1, kMathThreads);

    // output carried to the next step (Z_n is finished after the next barrier)
    float zprev[2][4] = {}, qprev[2][4] = {};
    int zprev_n = -1;

    auto finish_z = [&](int n, int par_stats) {
        // zprev holds Zbar_n^T; write Z_n (bf16) into the staging ring
        float z[2][4];
        if (LN) {
            // per-token mean / rstd from the exchanged partial sums
            const int tk = g >> 1, q = g & 1;
            const int t = 8 * (tk >> 1) + 2 * c + (tk & 1);
            const float4 w4 = *reinterpret_cast<const float4 *>(s.zred[par_stats][t][q]);
            float tot = (w4.x + w4.y) + (w4.z + w4.w);
            float oth = __shfl_xor_sync(0xffffffffu, tot, 4);
            const float s1 = q ? oth : tot, s2 = q ? tot : oth;
            const float mu = s1 * (1.f / D);
            const float var = fmaxf(s2 * (1.f / D) - mu * mu, 0.f);
            const float r = rsqrtf(var + p.eps);
#pragma unroll
            for (int tq = 0; tq < 4; ++tq) {
                const float m_t = __shfl_sync(0xffffffffu, mu, c + 8 * tq);
                const float r_t = __shfl_sync(0xffffffffu, r, c + 8 * tq);
                const int u = tq >> 1, e = tq & 1;
                z[u][e] = qprev[u][e] + fmaf(ga0 * (zprev[u][e] - m_t), r_t, be0);
                z[u][2 + e] = qprev[u][2 + e] + fmaf(ga1 * (zprev[u][2 + e] - m_t), r_t, be1);
            }
        } else {
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) z[u][i] = zprev[u][i];
        }
        uint32_t r[4];
        r[0] = ptx::pack_bf16(z[0][0], z[0][1]);
        r[1] = ptx::pack_bf16(z[0][2], z[0][3]);
        r[2] = ptx::pack_bf16(z[1][0], z[1][1]);
        r[3] = ptx::pack_bf16(z[1][2], z[1][3]);
        const int mrow = lane & 7, mat = lane >> 3;
        // matrices (j-block, t-block): (0,0), (1,0), (0,1), (1,1); stored rows = tokens
        const uint32_t zb = ptx::smem_addr(s.z[n % NZ]);
        ptx::stsm_x4_t(zb + ptx::sw128((mat >> 1) * 8 + mrow, warp * 2 + (mat & 1)), r);
        ptx::fence_proxy_async();
    };

    for (int n = 0; n < N; ++n) {
        const int par = n & 1;
        if (n + 2 < N && (n + 2) % TPS == 0) wait_stage((n + 2) / TPS);

        // (1) products from W_n: next key tile (lookahead) and this query tile
        float xacc[2][4], yacc[2][4];
        if (n + 1 < N) product(xacc, s.k, n + 1);
        product(yacc, s.q, n);
        // (2) input-only blocks for mini-batch n + 1
        if (n + 1 < N) compute_sfrag(n + 1, (n + 1) % 3);

        // (3) G_n from P_n
        float gmat[2][4];
        float vt[2][4];
        load_T(vt, s.v, n);
        float qt[2][4];
        load_T(qt, s.q, n);
        if (LN) {
            float kt[2][4];
            load_T(kt, s.k, n);
            // b'_j = beta_j - (v - k); gb = gamma * b'
            float gb[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                gb[u][0] = ga0 * (be0 - vt[u][0] + kt[u][0]);
                gb[u][1] = ga0 * (be0 - vt[u][1] + kt[u][1]);
                gb[u][2] = ga1 * (be1 - vt[u][2] + kt[u][2]);
                gb[u][3] = ga1 * (be1 - vt[u][3] + kt[u][3]);
            }
            const float g20 = ga0 * ga0, g21 = ga1 * ga1;
            // per-token partial sums over this thread's two features
            float vs[24];
#pragma unroll
            for (int tk = 0; tk < 4; ++tk) {
                const int u = tk >> 1, e = tk & 1;
                const float z0 = pacc[u][e], z1 = pacc[u][2 + e];
                const float a0 = g20 * z0, a1 = g21 * z1;
                vs[tk * 6 + 0] = z0 + z1;
                vs[tk * 6 + 1] = fmaf(z0, z0, z1 * z1);
                vs[tk * 6 + 2] = a0 + a1;
                vs[tk * 6 + 3] = fmaf(a0, z0, a1 * z1);
                vs[tk * 6 + 4] = fmaf(gb[u][e], z0, gb[u][2 + e] * z1);
                vs[tk * 6 + 5] = gb[u][e] + gb[u][2 + e];
            }
            // reduce-scatter over the 8 lanes sharing c (lane bits 4, 3, 2)
            float a12[12];
            {
                const bool hi = (lane >> 4) & 1;
#pragma unroll
                for (int i = 0; i < 12; ++i) {
                    const float snd = hi ? vs[i] : vs[12 + i];
                    const float kp = hi ? vs[12 + i] : vs[i];
                    a12[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 16);
                }
            }
            float a6[6];
            {
                const bool hi = (lane >> 3) & 1;
#pragma unroll
                for (int i = 0; i < 6; ++i) {
                    const float snd = hi ? a12[i] : a12[6 + i];
                    const float kp = hi ? a12[6 + i] : a12[i];
                    a6[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 8);
                }
            }
            float a3[3];
            {
                const bool hi = (lane >> 2) & 1;
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const float snd = hi ? a6[i] : a6[3 + i];
                    const float kp = hi ? a6[3 + i] : a6[i];
                    a3[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 4);
                }
            }
            // lane holds token tk = g/2, quantities 3 (g & 1) + 0..2
            const int tk = g >> 1, qh = g & 1;
            const int t = 8 * (tk >> 1) + 2 * c + (tk & 1);
#pragma unroll
            for (int i = 0; i < 3; ++i) s.red[par][t][3 * qh + i][warp] = a3[i];
            // Zbar stats of the previous step ride on the same barrier
            if (zprev_n >= 0) {
                float zs[8];
#pragma unroll
                for (int tq = 0; tq < 4; ++tq) {
                    const int u = tq >> 1, e = tq & 1;
                    const float z0 = zprev[u][e], z1 = zprev[u][2 + e];
                    zs[tq * 2 + 0] = z0 + z1;
                    zs[tq * 2 + 1] = fmaf(z0, z0, z1 * z1);
                }
                float b4[4];
                {
                    const bool hi = (lane >> 4) & 1;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float snd = hi ? zs[i] : zs[4 + i];
                        const float kp = hi ? zs[4 + i] : zs[i];
                        b4[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 16);
                    }
                }
                float b2[2];
                {
                    const bool hi = (lane >> 3) & 1;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const float snd = hi ? b4[i] : b4[2 + i];
                        const float kp = hi ? b4[2 + i] : b4[i];
                        b2[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 8);
                    }
                }
                const bool hi = (lane >> 2) & 1;
                const float snd = hi ? b2[0] : b2[1];
                const float kp = hi ? b2[1] : b2[0];
                const float b1 = kp + __shfl_xor_sync(0xffffffffu, snd, 4);
                // lane holds token g/2 (same t as above), quantity g & 1
                s.zred[par][t][qh][warp] = b1;
            }
            if (warp == 0 && lane == 0) ptx::bulk_wait_read<NZ - 2>();
            ptx::named_bar(1, kMathThreads);
            // totals for (t, 3 qh + i), then the partner lane supplies the other three
            float tot[3];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const float4 w4 = *reinterpret_cast<const float4 *>(s.red[par][t][3 * qh + i]);
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
            // G_j = (z - mu) (r^2 gamma_j^2 - r^2 m2) + r gamma_j b'_j - r m1
#pragma unroll
            for (int tq = 0; tq < 4; ++tq) {
                const int src = c + 8 * tq;
                const float mu_t = __shfl_sync(0xffffffffu, mu, src);
                const float a_t = __shfl_sync(0xffffffffu, co_a, src);
                const float b_t = __shfl_sync(0xffffffffu, co_b, src);
                const float r_t = __shfl_sync(0xffffffffu, r, src);
                const float e_t = __shfl_sync(0xffffffffu, co_e, src);
                const int u = tq >> 1, e = tq & 1;
                const float zc0 = pacc[u][e] - mu_t, zc1 = pacc[u][2 + e] - mu_t;
                gmat[u][e] = fmaf(zc0, fmaf(a_t, g20, -b_t), fmaf(r_t, gb[u][e], -e_t));
                gmat[u][2 + e] = fmaf(zc1, fmaf(a_t, g21, -b_t), fmaf(r_t, gb[u][2 + e], -e_t));
            }
        } else {
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) gmat[u][i] = pacc[u][i] - vt[u][i];
            if (warp == 0 && lane == 0) ptx::bulk_wait_read<NZ - 2>();
            ptx::named_bar(1, kMathThreads);
        }

        // the barrier above also published the block fragments of step n; issue
        // the previous output (its tile is complete) and finish Z_{n-1}
        if (zprev_n >= 0) finish_z(zprev_n, par);
        if (n >= 2 && warp == 0 && lane == 0) {
            // Z_{n-2} was finished before this step's barrier
            ptx::tma_store_3d(&tmZ, ptx::smem_addr(s.z[(n - 2) % NZ]), 0, (n - 2) * MB, bh);
            ptx::bulk_commit();
        }
        // release the stage whose last mini-batch was n - 1
        if (n >= 1 && (n % TPS) == 0 && warp == 0 && lane == 0)
            ptx::mbar_arrive(ptx::smem_addr(&s.empty[((n / TPS) - 1) % NSS]));

        // (4) -G and -eta G as A fragments (rows = features, k = tokens)
        const int s0 = 2 * c;
        const float e00 = eta_at(n, s0), e01 = eta_at(n, s0 + 1);
        const float e10 = eta_at(n, s0 + 8), e11 = eta_at(n, s0 + 9);
        uint32_t ng[4], nge[4];
        ng[0] = ptx::pack_bf16(-gmat[0][0], -gmat[0][1]);
        ng[1] = ptx::pack_bf16(-gmat[0][2], -gmat[0][3]);
        ng[2] = ptx::pack_bf16(-gmat[1][0], -gmat[1][1]);
        ng[3] = ptx::pack_bf16(-gmat[1][2], -gmat[1][3]);
        nge[0] = ptx::pack_bf16(-e00 * gmat[0][0], -e01 * gmat[0][1]);
        nge[1] = ptx::pack_bf16(-e00 * gmat[0][2], -e01 * gmat[0][3]);
        nge[2] = ptx::pack_bf16(-e10 * gmat[1][0], -e11 * gmat[1][1]);
        nge[3] = ptx::pack_bf16(-e10 * gmat[1][2], -e11 * gmat[1][3]);

        // (5) chain: P_{n+1} = X_{n+1} - G_n^T M^T;  output: Zbar_n = Y_n - G_n^T B^T
        uint32_t bf[2][2];
        if (n + 1 < N) {
            read_sfrag(n % 3, 0, bf);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
#pragma unroll
                for (int i = 0; i < 4; ++i) pacc[u][i] = xacc[u][i];
                ptx::mma_bf16(pacc[u], ng, bf[u][0], bf[u][1]);
            }
        }
        read_sfrag(n % 3, 1, bf);
#pragma unroll
        for (int u = 0; u < 2; ++u) ptx::mma_bf16(yacc[u], ng, bf[u][0], bf[u][1]);

        // (6) state update: W^T += (-eta G)^T K_n, c -= eta^T G
        {
            const int mrow = lane & 7, mat = lane >> 3;
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                // matrices (s-block, i-chunk): (0, 2pp), (1, 2pp), (0, 2pp+1), (1, 2pp+1)
                uint32_t r[4];
                ptx::ldsm_x4_t(tile_addr(s.k, n, (mat & 1) * 8 + mrow, 2 * pp + (mat >> 1)), r);
                ptx::mma_bf16(wt[2 * pp], nge, r[0], r[1]);
                ptx::mma_bf16(wt[2 * pp + 1], nge, r[2], r[3]);
            }
            pack_w();
            float d0 = e00 * gmat[0][0] + e01 * gmat[0][1] + e10 * gmat[1][0] + e11 * gmat[1][1];
            float d1 = e00 * gmat[0][2] + e01 * gmat[0][3] + e10 * gmat[1][2] + e11 * gmat[1][3];
            d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
            d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
            cb0 -= d0;
            cb1 -= d1;
        }

        // (7) keep Zbar_n and Q_n for the next step's output stage
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                zprev[u][i] = yacc[u][i];
                qprev[u][i] = qt[u][i];
            }
        zprev_n = n;
    }

    // ---- tail: last output, final stores, final state
    {
        const int par = N & 1;
        if (LN) {
            float zs[8];
#pragma unroll
            for (int tq = 0; tq < 4; ++tq) {
                const int u = tq >> 1, e = tq & 1;
                const float z0 = zprev[u][e], z1 = zprev[u][2 + e];
                zs[tq * 2 + 0] = z0 + z1;
                zs[tq * 2 + 1] = fmaf(z0, z0, z1 * z1);
            }
            float b4[4];
            {
                const bool hi = (lane >> 4) & 1;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float snd = hi ? zs[i] : zs[4 + i];
                    const float kp = hi ? zs[4 + i] : zs[i];
                    b4[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 16);
                }
            }
            float b2[2];
            {
                const bool hi = (lane >> 3) & 1;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float snd = hi ? b4[i] : b4[2 + i];
                    const float kp = hi ? b4[2 + i] : b4[i];
                    b2[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 8);
                }
            }
            const bool hi = (lane >> 2) & 1;
            const float snd = hi ? b2[0] : b2[1];
            const float kp = hi ? b2[1] : b2[0];
            const float b1 = kp + __shfl_xor_sync(0xffffffffu, snd, 4);
            const int tk = g >> 1;
            const int t = 8 * (tk >> 1) + 2 * c + (tk & 1);
            s.zred[par][t][g & 1][warp] = b1;
        }
        if (warp == 0 && lane == 0) ptx::bulk_wait_read<NZ - 2>();
        ptx::named_bar(1, kMathThreads);
        finish_z(N - 1, par);
        ptx::named_bar(1, kMathThreads);
        if (warp == 0 && lane == 0) {
            for (int n = max(0, N - 2); n < N; ++n) {
                ptx::tma_store_3d(&tmZ, ptx::smem_addr(s.z[n % NZ]), 0, n * MB, bh);
                ptx::bulk_commit();
            }
            ptx::bulk_wait<0>();
        }
    }
    {
        float *Wf = p.Wf + (size_t)bh * D * D;
#pragma unroll
        for (int pt = 0; pt < 8; ++pt) {
            const int i = pt * 8 + 2 * c;
            Wf[i * D + j0] = wt[pt][0];
            Wf[(i + 1) * D + j0] = wt[pt][1];
            Wf[i * D + j1] = wt[pt][2];
            Wf[(i + 1) * D + j1] = wt[pt][3];
        }
        if (c == 0) {
            p.bf[(size_t)bh * D + j0] = cb0;
            p.bf[(size_t)bh * D + j1] = cb1;
        }
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode()
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

// [BH][L][64] bf16 viewed as a 3-D tensor; boxes of `rows` tokens, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, int L, int BH, int rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

long long g_wait_ns = kDefaultWaitNs;
int g_withhold_loads = 0;

}  // namespace

void set_wait_timeout_ns(long long ns) { g_wait_ns = ns > 0 ? ns : kDefaultWaitNs; }
void set_withhold_loads(int on) { g_withhold_loads = on != 0; }

bool linear_tc_supported(const ttt_desc &d)
{
    return d.io_dtype == TTT_BF16 && d.d == D && d.mini_batch == MB;
}

cudaError_t launch_linear_tc(const LinearArgs &a)
{
    const ttt_desc &d = a.desc;
    const int BH = d.B * d.H;
    CUtensorMap mq, mk, mv, mz;
    if (!make_map(&mq, a.Q, d.L, BH, ST) || !make_map(&mk, a.K, d.L, BH, ST) ||
        !make_map(&mv, a.V, d.L, BH, ST) || !make_map(&mz, a.Z, d.L, BH, MB))
        return cudaErrorInvalidValue;
    Params p{d.H, d.L, d.residual_ln, d.ln_eps, g_wait_ns, g_withhold_loads, a.eta, a.W0, a.b0, a.gamma, a.beta,
             a.W_final, a.b_final, a.status, d.init_per_batch};
    const size_t smem = sizeof(Smem) + 1024;
    auto kern = d.residual_ln ? linear_fused_kernel<true> : linear_fused_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<BH, kThreads, smem, a.stream>>>(mq, mk, mv, mz, p);
    return cudaGetLastError();
}

}  // namespace ttt
