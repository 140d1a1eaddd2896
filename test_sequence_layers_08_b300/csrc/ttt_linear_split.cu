// ttt_linear_split.cu -- fused TTT-Linear forward, bf16 I/O, d = 64, b = 16, with the work of
// one (batch, head) split between two kinds of warps so that the sequential part of the scan
// has warps of its own.
//
// The method (damodev.csdn.net TTT article, sections 3.1 and 4.1-4.2; residual LayerNorm of
// the lryc.cn TTT article, section 2.1), per (batch, head) and mini-batch n of 16 tokens:
//   P_n = K_n W_n + 1 c_n,   G_n = P_n - V_n  or  LNbwd(P_n; V_n - K_n)
//   W_{n+1} = W_n - K_n^T diag(eta_n) G_n,   c_{n+1} = c_n - eta_n^T G_n
//   Z_n = f_out(Q_n W_n + 1 c_n - (tril(Q_n K_n^T + 1) diag(eta_n)) G_n)
// With M(m, n) = (K_m K_n^T + 1) diag(eta_n) (16 x 16, inputs only), the key-side product is
// re-associated exactly two mini-batches back:
//   P_{n+1} = X_{n+1} - M(n+1, n-1) G_{n-1} - M(n+1, n) G_n,   X_{n+1} = K_{n+1} W_{n-1} + 1 c_{n-1}
// so the only sequential chain is G_n -> one 16 x 16 x 16 product -> P_{n+1} -> G_{n+1}, and
// everything that needs the state W has two mini-batches of slack.
//
// B300 design: one CTA per (batch, head), eight warps, two per SM sub-partition.
//   * chain warps 0-3 (warp w owns output features 16w..16w+15): the LayerNorm backward of
//     P_n, G_n, the two 16 x 16 chain products and the bias increment eta^T G.  They read
//     nothing from global memory or the stage ring: everything arrives through hand-off rings.
//   * state warps 4-7 (warp w + 4 owns the same 16 features as chain warp w): W^T in registers
//     (fp32 warp-MMA accumulators), its update, the d x d products X_{n+3} = K_{n+3} W_{n+1} and
//     Y_{n+1} = Q_{n+1} W_{n+1}, the input-only 16 x 16 blocks, the residual-LayerNorm inputs
//     gamma (beta - v + k) of the chain, the output (Y_n - tril-block G_n, LayerNorm, + Q_n)
//     and the Z stores; they own the TMA stage ring of Q, K, V, eta.
//   * hand-offs are thread to thread (chain thread (w, lane) <-> state thread (w + 4, lane)
//     hold the same features in the same fragment layout) through 4-deep shared-memory rings,
//     each slot guarded by a full and an empty mbarrier (phase-tracked, bounded waits).
//   * every contraction is a bf16 m16n8k16 warp MMA with fp32 accumulation; the LayerNorm
//     statistics are fp32 (one-pass sums on a bias shifted by its mean, which LayerNorm does
//     not see).
// Every mbarrier wait is bounded; a wait that runs out sets the library's failure flag, and
// from then on no warp of the CTA waits again (results are then unspecified).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int D = 64;           // head dim
constexpr int MB = 16;          // mini-batch
constexpr int ST = 64;          // tokens per stage
constexpr int TPS = ST / MB;    // mini-batches per stage
constexpr int NSS = 6;          // stages in the ring
constexpr int NZ = 4;           // Z staging tiles
constexpr int R = 4;            // hand-off ring depth
constexpr int kThreads = 256;
constexpr uint32_t kStageTileBytes = ST * D * 2;
constexpr int kBarChain = 1, kBarState = 2;   // named barriers (128 threads each)
constexpr long long kDrainNs = 1000000000ll;

struct __align__(1024) Smem {
    __nv_bfloat16 q[NSS][ST * D];
    __nv_bfloat16 k[NSS][ST * D];
    __nv_bfloat16 v[NSS][ST * D];
    __nv_bfloat16 z[NZ][MB * D];
    float eta[NSS][ST];
    // chain -> state: -G_n as bf16 A fragments, and the bias increment eta^T G_n
    uint4 hg[R][4][32];
    float2 hc[R][4][32];
    // state -> chain: X_m = K_m W_{m-2} + c_{m-2} as fp32 C fragments
    float4 hx[R][4][32][2];
    // state -> chain, inputs of chain step m: gamma (beta - v + k) (or -v), eta_m, and the
    // blocks M(m+1, m) (next) and M(m+1, m-1) (prev) as B fragments of the chain product
    float4 hgb[R][4][32][2];
    float heta[R][MB];
    uint4 hmc[R][2][32];
    // state warps: the output block eta_s (Q_n[t] . K_n[s] + 1) [s <= t] by parity of n
    uint4 hmo[2][32];
    float red[2][MB][36];      // chain LayerNorm exchange: six sums x four warps (padded)
    float zred[2][MB][12];     // output LayerNorm exchange: two sums x four warps (padded)
    unsigned long long full[NSS];
    unsigned long long g_full[R][4], g_empty[R][4], x_full[R][4], x_empty[R][4];
    unsigned long long in_full[R], in_empty[R];
    int abort_flag;
};

static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared-memory layout exceeds the per-CTA limit");

struct Params {
    int H, L;
    float eps;
    long long wait_ns;
    int withhold_loads;
    const float *eta, *W0, *b0, *gamma, *beta;
    float *Wf, *bf;
    unsigned int *status;
    int init_per_batch;
    int hoff = 0;            // head index of row 0 of this call
};

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, long long limit, int *abort_flag,
                                       unsigned int *status)
{
    if (*(volatile int *)abort_flag) return false;
    if (ptx::mbar_wait_bounded(bar, parity, limit)) return true;
    *(volatile int *)abort_flag = 1;
    atomicOr(status, kStatusTimeout);
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

template <bool LN>
__global__ void __launch_bounds__(kThreads, 1)
linear_split_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmZ,
                    Params p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    Smem &s = *reinterpret_cast<Smem *>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3;                 // feature block of this warp (both roles)
    const bool chain = warp < 4;
    const int bh = blockIdx.x, h = (p.hoff + bh) % p.H;
    const int N = p.L / MB;
    const int NST = (p.L + ST - 1) / ST;
    const int g = lane >> 2, c = lane & 3, mrow = lane & 7, mat = lane >> 3;
    const int j0 = wq * 16 + g, j1 = j0 + 8;   // this thread's two features
    constexpr int kIssuer = 128;             // state warp 4, lane 0: stage copies, Z stores

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
    const int nissue = p.withhold_loads ? 0 : NST;
    int issued = min(NSS, nissue);
    if (tid == 0) {
        for (int i = 0; i < NSS; ++i) ptx::mbar_init(ptx::smem_addr(&s.full[i]), 1);
        for (int r = 0; r < R; ++r) {
            for (int w = 0; w < 4; ++w) {
                ptx::mbar_init(ptx::smem_addr(&s.g_full[r][w]), 1);
                ptx::mbar_init(ptx::smem_addr(&s.g_empty[r][w]), 1);
                ptx::mbar_init(ptx::smem_addr(&s.x_full[r][w]), 1);
                ptx::mbar_init(ptx::smem_addr(&s.x_empty[r][w]), 1);
            }
            ptx::mbar_init(ptx::smem_addr(&s.in_full[r]), 4);
            ptx::mbar_init(ptx::smem_addr(&s.in_empty[r]), 4);
        }
        s.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (tid == kIssuer) {
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmZ);
    }
    __syncthreads();
    if (tid == kIssuer)
        for (int st = 0; st < issued; ++st) issue_stage(st);

    bool aborted = false;
    // bounded wait for phase `parity` of the mbarrier at shared address `bar`
    auto wait_bar = [&](uint32_t bar, uint32_t parity) {
        if (aborted) return;
        if (ptx::mbar_try_wait(bar, parity)) return;
        aborted = !wait_slow(bar, parity, p.wait_ns, &s.abort_flag, p.status);
    };
    // the k-th use (k = m / R) of ring slot m % R waits for phase parity k & 1 of its full
    // barrier; the producer of use k >= 1 waits for phase (k - 1) & 1 of its empty barrier
    auto par_full = [](int m) -> uint32_t { return (uint32_t)((m / R) & 1); };
    auto par_empty = [](int m) -> uint32_t { return (uint32_t)((m / R - 1) & 1); };

    if (chain) {
        // =============================================================== chain warps
        float pacc[2][4];                     // P_n: rows = features j0/j1, cols = tokens
        uint32_t ngprev[4] = {0u, 0u, 0u, 0u};  // -G_{n-1} as A fragments
        const int tk = g >> 1, qh = g & 1;
        const int t_own = 8 * (tk >> 1) + 2 * c + (tk & 1);
        float ga0 = 1.f, ga1 = 1.f, C1 = 0.f;
        if (LN) {
            ga0 = p.gamma[(size_t)h * D + j0];
            ga1 = p.gamma[(size_t)h * D + j1];
            float part = ga0 * ga0 + ga1 * ga1;
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) s.red[0][0][warp] = part;
            ptx::named_bar(kBarChain, 128);
            const float4 w4 = *reinterpret_cast<const float4 *>(s.red[0][0]);
            C1 = (w4.x + w4.y) + (w4.z + w4.w);
            ptx::named_bar(kBarChain, 128);
        }
        const float g20 = ga0 * ga0, g21 = ga1 * ga1;

        // P_0 = X_0 (slot 0)
        {
            wait_bar(ptx::smem_addr(&s.x_full[0][wq]), 0);
            const float4 a = s.hx[0][wq][lane][0], b = s.hx[0][wq][lane][1];
            pacc[0][0] = a.x; pacc[0][1] = a.y; pacc[0][2] = a.z; pacc[0][3] = a.w;
            pacc[1][0] = b.x; pacc[1][1] = b.y; pacc[1][2] = b.z; pacc[1][3] = b.w;
            __syncwarp();
            if (lane == 0) mbar_arrive(ptx::smem_addr(&s.x_empty[0][wq]));
        }

        for (int n = 0; n < N; ++n) {
            const int par = n & 1;
            const bool more = n + 1 < N;      // there is a P_{n+1} to form
            // ---- inputs of this step
            const int si = n % R;
            wait_bar(ptx::smem_addr(&s.in_full[si]), par_full(n));
            float gb[2][4];
            {
                const float4 a = s.hgb[si][wq][lane][0], b = s.hgb[si][wq][lane][1];
                gb[0][0] = a.x; gb[0][1] = a.y; gb[0][2] = a.z; gb[0][3] = a.w;
                gb[1][0] = b.x; gb[1][1] = b.y; gb[1][2] = b.z; gb[1][3] = b.w;
            }
            const float2 e01 = *reinterpret_cast<const float2 *>(&s.heta[si][2 * c]);
            const float2 e89 = *reinterpret_cast<const float2 *>(&s.heta[si][2 * c + 8]);
            const uint4 mnext = s.hmc[si][0][lane], mprev = s.hmc[si][1][lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(ptx::smem_addr(&s.in_empty[si]));

            // ---- early part of P_{n+1}: X_{n+1} - M(n+1, n-1) G_{n-1} (off the chain)
            float xp[2][4];
            if (more) {
                const int sx = (n + 1) % R;
                wait_bar(ptx::smem_addr(&s.x_full[sx][wq]), par_full(n + 1));
                const float4 a = s.hx[sx][wq][lane][0], b = s.hx[sx][wq][lane][1];
                xp[0][0] = a.x; xp[0][1] = a.y; xp[0][2] = a.z; xp[0][3] = a.w;
                xp[1][0] = b.x; xp[1][1] = b.y; xp[1][2] = b.z; xp[1][3] = b.w;
                __syncwarp();
                if (lane == 0) mbar_arrive(ptx::smem_addr(&s.x_empty[sx][wq]));
                if (n > 0) {
                    ptx::mma_bf16(xp[0], ngprev, mprev.x, mprev.z);
                    ptx::mma_bf16(xp[1], ngprev, mprev.y, mprev.w);
                }
            }

            // ---- G_n
            float gmat[2][4];
            if (LN) {
                float vs[24];
#pragma unroll
                for (int t4 = 0; t4 < 4; ++t4) {
                    const int u = t4 >> 1, e = t4 & 1;
                    const float z0 = pacc[u][e], z1 = pacc[u][2 + e];
                    const float a0 = g20 * z0, a1 = g21 * z1;
                    vs[t4 * 6 + 0] = z0 + z1;
                    vs[t4 * 6 + 1] = fmaf(z0, z0, z1 * z1);
                    vs[t4 * 6 + 2] = a0 + a1;
                    vs[t4 * 6 + 3] = fmaf(a0, z0, a1 * z1);
                    vs[t4 * 6 + 4] = fmaf(gb[u][e], z0, gb[u][2 + e] * z1);
                    vs[t4 * 6 + 5] = gb[u][e] + gb[u][2 + e];
                }
                // reduce-scatter over the 8 lanes sharing c (lane bits 4, 3, 2)
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
                for (int i = 0; i < 3; ++i) s.red[par][t_own][4 * (3 * qh + i) + wq] = a3[i];
                ptx::named_bar(kBarChain, 128);
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
                    const float zc0 = pacc[u][e] - mu_t, zc1 = pacc[u][2 + e] - mu_t;
                    gmat[u][e] = fmaf(zc0, fmaf(a_t, g20, -b_t), fmaf(r_t, gb[u][e], -e_t));
                    gmat[u][2 + e] = fmaf(zc1, fmaf(a_t, g21, -b_t), fmaf(r_t, gb[u][2 + e], -e_t));
                }
            } else {
                // gb holds -V_n
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) gmat[u][i] = pacc[u][i] + gb[u][i];
            }

            // ---- -G_n as A fragments; P_{n+1} = xp - M(n+1, n) G_n
            uint32_t ng[4];
            ng[0] = ptx::pack_bf16(-gmat[0][0], -gmat[0][1]);
            ng[1] = ptx::pack_bf16(-gmat[0][2], -gmat[0][3]);
            ng[2] = ptx::pack_bf16(-gmat[1][0], -gmat[1][1]);
            ng[3] = ptx::pack_bf16(-gmat[1][2], -gmat[1][3]);
            if (more) {
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) pacc[u][i] = xp[u][i];
                ptx::mma_bf16(pacc[0], ng, mnext.x, mnext.z);
                ptx::mma_bf16(pacc[1], ng, mnext.y, mnext.w);
            }
            // bias increment eta^T G_n over this thread's tokens, then the quad
            float d0 = e01.x * gmat[0][0] + e01.y * gmat[0][1] + e89.x * gmat[1][0] + e89.y * gmat[1][1];
            float d1 = e01.x * gmat[0][2] + e01.y * gmat[0][3] + e89.x * gmat[1][2] + e89.y * gmat[1][3];
            d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
            d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
            // ---- hand G_n to the state warp
            {
                const int sg = n % R;
                if (n >= R) wait_bar(ptx::smem_addr(&s.g_empty[sg][wq]), par_empty(n));
                s.hg[sg][wq][lane] = make_uint4(ng[0], ng[1], ng[2], ng[3]);
                s.hc[sg][wq][lane] = make_float2(d0, d1);
                __syncwarp();
                if (lane == 0) mbar_arrive(ptx::smem_addr(&s.g_full[sg][wq]));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) ngprev[i] = ng[i];
        }
        return;
    }

    // =================================================================== state warps
    const int sw = wq;   // 0..3 among the state warps
    auto wait_stage = [&](int st) { wait_bar(ptx::smem_addr(&s.full[st % NSS]), (uint32_t)((st / NSS) & 1)); };
    auto tile_addr = [&](const __nv_bfloat16 (*arr)[ST * D], int n, int t, int chunk) -> uint32_t {
        const uint32_t toff = (uint32_t)(((n / TPS) % NSS) * (ST * D * 2) + (n % TPS) * (MB * 128));
        return ptx::smem_addr(arr[0]) + toff + (uint32_t)(t * 128 + ((chunk ^ mrow) << 4));
    };
    auto eta_at = [&](int n, int t) -> float { return s.eta[(n / TPS) % NSS][(n % TPS) * MB + t]; };

    // initial state: W^T rows j0/j1 as fp32 accumulators, c (shifted by its mean with LN)
    float wt[8][4];
    const size_t init = p.init_per_batch ? (size_t)bh : (size_t)h;
    {
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
    float cb0 = p.b0[init * D + j0];
    float cb1 = p.b0[init * D + j1];
    float ga0 = 1.f, ga1 = 1.f, be0 = 0.f, be1 = 0.f, pivot = 0.f;
    if (LN) {
        ga0 = p.gamma[(size_t)h * D + j0];
        ga1 = p.gamma[(size_t)h * D + j1];
        be0 = p.beta[(size_t)h * D + j0];
        be1 = p.beta[(size_t)h * D + j1];
        // LayerNorm pivot: the scan runs on c - mean(b0) (LN and its backward do not see a
        // common shift of P or of the output's pre-activation); the mean goes back into b_final
        float pb = cb0 + cb1;
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) pb += __shfl_xor_sync(0xffffffffu, pb, o);
        if (lane == 0) s.zred[0][0][sw] = pb;
        ptx::named_bar(kBarState, 128);
        const float4 p4 = *reinterpret_cast<const float4 *>(s.zred[0][0]);
        pivot = ((p4.x + p4.y) + (p4.z + p4.w)) * (1.f / D);
        cb0 -= pivot;
        cb1 -= pivot;
        ptx::named_bar(kBarState, 128);
    }

    uint32_t wa[4][4];
    auto pack_w = [&]() {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            wa[q][0] = ptx::pack_bf16(wt[2 * q][0], wt[2 * q][1]);
            wa[q][1] = ptx::pack_bf16(wt[2 * q][2], wt[2 * q][3]);
            wa[q][2] = ptx::pack_bf16(wt[2 * q + 1][0], wt[2 * q + 1][1]);
            wa[q][3] = ptx::pack_bf16(wt[2 * q + 1][2], wt[2 * q + 1][3]);
        }
    };
    // acc = W^T X^T + c for the 16-token tile X of mini-batch n
    auto product = [&](float (*acc)[4], const __nv_bfloat16 (*arr)[ST * D], int n) {
        uint32_t r[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            ptx::ldsm_x4(tile_addr(arr, n, (mat >> 1) * 8 + mrow, 2 * q + (mat & 1)), r[q]);
        float hi[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            acc[u][0] = cb0; acc[u][1] = cb0; acc[u][2] = cb1; acc[u][3] = cb1;
            hi[u][0] = 0.f; hi[u][1] = 0.f; hi[u][2] = 0.f; hi[u][3] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            ptx::mma_bf16(acc[0], wa[q], r[q][0], r[q][1]);
            ptx::mma_bf16(acc[1], wa[q], r[q][2], r[q][3]);
            ptx::mma_bf16(hi[0], wa[q + 2], r[q + 2][0], r[q + 2][1]);
            ptx::mma_bf16(hi[1], wa[q + 2], r[q + 2][2], r[q + 2][3]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[u][i] += hi[u][i];
    };
    // C-fragment layout (rows = features j0/j1, cols = tokens) of a bf16 tile, transposed
    auto load_T = [&](float (*out)[4], const __nv_bfloat16 (*arr)[ST * D], int n) {
        uint32_t r[4];
        ptx::ldsm_x4_t(tile_addr(arr, n, (mat >> 1) * 8 + mrow, sw * 2 + (mat & 1)), r);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            out[u][0] = ptx::bf16_lo(r[2 * u]);
            out[u][1] = ptx::bf16_hi(r[2 * u]);
            out[u][2] = ptx::bf16_lo(r[2 * u + 1]);
            out[u][3] = ptx::bf16_hi(r[2 * u + 1]);
        }
    };
    // half `half` (source tokens s in [8 half, 8 half + 8)) of the block
    //   eta_{ns}[s] (A_{na}[t] . K_{ns}[s] + 1)  (masked to s <= t when causal)
    // as the B-fragment pair of the chain / output product, for target tile A_{na}
    auto gram_half = [&](const __nv_bfloat16 (*A)[ST * D], int na, int ns, int half, bool causal) -> uint2 {
        uint32_t a[4][4], b[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            ptx::ldsm_x4(tile_addr(A, na, (mat & 1) * 8 + mrow, 2 * q + (mat >> 1)), a[q]);
            ptx::ldsm_x4(tile_addr(s.k, ns, half * 8 + mrow, 2 * q + (mat & 1)), b[q]);
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, ac2[4] = {0.f, 0.f, 0.f, 0.f};
        ptx::mma_bf16(acc, a[0], b[0][0], b[0][1]);
        ptx::mma_bf16(ac2, a[2], b[2][0], b[2][1]);
        ptx::mma_bf16(acc, a[1], b[1][0], b[1][1]);
        ptx::mma_bf16(ac2, a[3], b[3][0], b[3][1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] += ac2[i];
        const int s0 = half * 8 + 2 * c;
        const float e0 = eta_at(ns, s0), e1 = eta_at(ns, s0 + 1);
        const float v0 = (causal && s0 > g) ? 0.f : e0 * (acc[0] + 1.f);
        const float v1 = (causal && s0 + 1 > g) ? 0.f : e1 * (acc[1] + 1.f);
        const float v2 = (causal && s0 > g + 8) ? 0.f : e0 * (acc[2] + 1.f);
        const float v3 = (causal && s0 + 1 > g + 8) ? 0.f : e1 * (acc[3] + 1.f);
        return make_uint2(ptx::pack_bf16(v0, v1), ptx::pack_bf16(v2, v3));
    };
    // inputs of chain step m (m + 1 < N gives the blocks; m = 0 has no "prev" block)
    auto produce_in = [&](int m) {
        const int si = m % R;
        if (m >= R) wait_bar(ptx::smem_addr(&s.in_empty[si]), par_empty(m));
        float gbv[2][4];
        if (LN) {
            float vt[2][4], kt[2][4];
            load_T(vt, s.v, m);
            load_T(kt, s.k, m);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                gbv[u][0] = ga0 * (be0 - vt[u][0] + kt[u][0]);
                gbv[u][1] = ga0 * (be0 - vt[u][1] + kt[u][1]);
                gbv[u][2] = ga1 * (be1 - vt[u][2] + kt[u][2]);
                gbv[u][3] = ga1 * (be1 - vt[u][3] + kt[u][3]);
            }
        } else {
            float vt[2][4];
            load_T(vt, s.v, m);
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) gbv[u][i] = -vt[u][i];
        }
        s.hgb[si][sw][lane][0] = make_float4(gbv[0][0], gbv[0][1], gbv[0][2], gbv[0][3]);
        s.hgb[si][sw][lane][1] = make_float4(gbv[1][0], gbv[1][1], gbv[1][2], gbv[1][3]);
        if (sw == 0 && lane < MB) s.heta[si][lane] = eta_at(m, lane);
        if (m + 1 < N) {
            // warp sw: block (sw >> 1) (0: next M(m+1, m), 1: prev M(m+1, m-1)), source half sw & 1
            const int which = sw >> 1, half = sw & 1;
            if (which == 0 || m > 0) {
                const uint2 f = gram_half(s.k, m + 1, which ? m - 1 : m, half, false);
                uint32_t *dst = reinterpret_cast<uint32_t *>(&s.hmc[si][which][lane]) + 2 * half;
                *reinterpret_cast<uint2 *>(dst) = f;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ptx::smem_addr(&s.in_full[si]));
    };
    auto produce_x = [&](int m) {   // X_m = K_m W + c with the current (packed) W
        const int sx = m % R;
        float xa[2][4];
        product(xa, s.k, m);
        if (m >= R) wait_bar(ptx::smem_addr(&s.x_empty[sx][sw]), par_empty(m));
        s.hx[sx][sw][lane][0] = make_float4(xa[0][0], xa[0][1], xa[0][2], xa[0][3]);
        s.hx[sx][sw][lane][1] = make_float4(xa[1][0], xa[1][1], xa[1][2], xa[1][3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(ptx::smem_addr(&s.x_full[sx][sw]));
    };
    auto produce_mo = [&](int m) {   // output block of mini-batch m, warps 0 and 1 (halves)
        if (sw < 2) {
            const uint2 f = gram_half(s.q, m, m, sw, true);
            uint32_t *dst = reinterpret_cast<uint32_t *>(&s.hmo[m & 1][lane]) + 2 * sw;
            *reinterpret_cast<uint2 *>(dst) = f;
        }
    };

    // reduce-scatter of 8 per-token values (4 tokens x 2 quantities) over the 8 lanes sharing c
    auto rs8 = [&](const float *zs) -> float {
        float b4[4], b2[2];
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
                b2[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 8);
            }
        }
        const bool hi = (lane >> 2) & 1;
        const float snd = hi ? b2[0] : b2[1];
        const float kp = hi ? b2[1] : b2[0];
        return kp + __shfl_xor_sync(0xffffffffu, snd, 4);
    };
    const int tk = g >> 1, qh = g & 1;
    const int t_own = 8 * (tk >> 1) + 2 * c + (tk & 1);

    // ---- prologue: stage 0, X_0 .. X_2 from W_0, Y_0, inputs of chain steps 0 and 1, M_out(0)
    wait_stage(0);
    pack_w();
    for (int m = 0; m < min(3, N); ++m) produce_x(m);
    float yprev[2][4];
    product(yprev, s.q, 0);
    produce_in(0);
    if (N > 1) produce_in(1);
    produce_mo(0);
    ptx::named_bar(kBarState, 128);   // M_out(0) is visible to every state warp

    for (int n = 0; n < N; ++n) {
        const int par = n & 1;
        // the inputs of this iteration reach mini-batch n + 3
        if ((n + 3) % TPS == 0 && n + 3 < N) wait_stage((n + 3) / TPS);
        // ---- input-only work, independent of G_n
        if (n + 2 < N) produce_in(n + 2);
        if (n + 1 < N) produce_mo(n + 1);
        float qt[2][4];
        load_T(qt, s.q, n);

        // ---- G_n from the chain warp
        uint4 ngv;
        float2 cd;
        {
            const int sg = n % R;
            wait_bar(ptx::smem_addr(&s.g_full[sg][sw]), par_full(n));
            ngv = s.hg[sg][sw][lane];
            cd = s.hc[sg][sw][lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(ptx::smem_addr(&s.g_empty[sg][sw]));
        }
        const uint32_t ng[4] = {ngv.x, ngv.y, ngv.z, ngv.w};

        // ---- output n: Zbar_n = Y_n - M_out(n) G_n, then Q_n + LN(Zbar_n)
        {
            const uint4 mo = s.hmo[n & 1][lane];
            ptx::mma_bf16(yprev[0], ng, mo.x, mo.z);
            ptx::mma_bf16(yprev[1], ng, mo.y, mo.w);
        }
        if (LN) {
            float zs[8];
#pragma unroll
            for (int tq = 0; tq < 4; ++tq) {
                const int u = tq >> 1, e = tq & 1;
                const float z0 = yprev[u][e], z1 = yprev[u][2 + e];
                zs[tq * 2 + 0] = z0 + z1;
                zs[tq * 2 + 1] = fmaf(z0, z0, z1 * z1);
            }
            s.zred[par][t_own][4 * qh + sw] = rs8(zs);
        }
        if (tid == kIssuer) ptx::bulk_wait_read<NZ - 2>();
        ptx::named_bar(kBarState, 128);
        // Z_{n-1} was finished before this barrier
        if (tid == kIssuer && n >= 1) {
            ptx::tma_store_3d(&tmZ, ptx::smem_addr(s.z[(n - 1) % NZ]), 0, (n - 1) * MB, bh);
            ptx::bulk_commit();
        }
        // the stage holding mini-batch n - 1 is no longer read: refill its slot
        if (tid == kIssuer && n >= TPS && n % TPS == 0 && n / TPS - 1 + NSS < nissue && !aborted) {
            ptx::fence_proxy_async();
            issue_stage(n / TPS - 1 + NSS);
            issued = n / TPS + NSS;
        }
        {
            float z[2][4];
            if (LN) {
                const float4 w4 = *reinterpret_cast<const float4 *>(&s.zred[par][t_own][4 * qh]);
                const float tot = (w4.x + w4.y) + (w4.z + w4.w);
                const float oth = __shfl_xor_sync(0xffffffffu, tot, 4);
                const float s1 = qh ? oth : tot, s2 = qh ? tot : oth;
                const float mu = s1 * (1.f / D);
                const float var = fmaxf(s2 * (1.f / D) - mu * mu, 0.f);
                const float r = rsqrtf(var + p.eps);
#pragma unroll
                for (int tq = 0; tq < 4; ++tq) {
                    const float m_t = __shfl_sync(0xffffffffu, mu, c + 8 * tq);
                    const float r_t = __shfl_sync(0xffffffffu, r, c + 8 * tq);
                    const int u = tq >> 1, e = tq & 1;
                    z[u][e] = qt[u][e] + fmaf(ga0 * (yprev[u][e] - m_t), r_t, be0);
                    z[u][2 + e] = qt[u][2 + e] + fmaf(ga1 * (yprev[u][2 + e] - m_t), r_t, be1);
                }
            } else {
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) z[u][i] = yprev[u][i];
            }
            uint32_t rr[4];
            rr[0] = ptx::pack_bf16(z[0][0], z[0][1]);
            rr[1] = ptx::pack_bf16(z[0][2], z[0][3]);
            rr[2] = ptx::pack_bf16(z[1][0], z[1][1]);
            rr[3] = ptx::pack_bf16(z[1][2], z[1][3]);
            const uint32_t zaddr = ptx::smem_addr(s.z[n % NZ]);
            ptx::stsm_x4_t(zaddr + ptx::sw128((mat >> 1) * 8 + mrow, sw * 2 + (mat & 1)), rr);
            ptx::fence_proxy_async();
        }

        // ---- W_{n+1} = W_n + (-eta G_n)^T K_n,  c_{n+1} = c_n - eta^T G_n
        {
            const int s0 = 2 * c;
            const float e00 = eta_at(n, s0), e01 = eta_at(n, s0 + 1);
            const float e10 = eta_at(n, s0 + 8), e11 = eta_at(n, s0 + 9);
            uint32_t nge[4];
            nge[0] = ptx::pack_bf16(e00 * ptx::bf16_lo(ng[0]), e01 * ptx::bf16_hi(ng[0]));
            nge[1] = ptx::pack_bf16(e00 * ptx::bf16_lo(ng[1]), e01 * ptx::bf16_hi(ng[1]));
            nge[2] = ptx::pack_bf16(e10 * ptx::bf16_lo(ng[2]), e11 * ptx::bf16_hi(ng[2]));
            nge[3] = ptx::pack_bf16(e10 * ptx::bf16_lo(ng[3]), e11 * ptx::bf16_hi(ng[3]));
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                uint32_t r[4];
                ptx::ldsm_x4_t(tile_addr(s.k, n, (mat & 1) * 8 + mrow, 2 * pp + (mat >> 1)), r);
                ptx::mma_bf16(wt[2 * pp], nge, r[0], r[1]);
                ptx::mma_bf16(wt[2 * pp + 1], nge, r[2], r[3]);
            }
            cb0 -= cd.x;
            cb1 -= cd.y;
        }
        // ---- products from W_{n+1}: X_{n+3} for the chain, Y_{n+1} for the next output
        if (n + 1 < N) {
            pack_w();
            if (n + 3 < N) produce_x(n + 3);
            product(yprev, s.q, n + 1);
        }
    }

    // ---- tail: the last Z tile, final state
    ptx::named_bar(kBarState, 128);
    if (tid == kIssuer) {
        ptx::tma_store_3d(&tmZ, ptx::smem_addr(s.z[(N - 1) % NZ]), 0, (N - 1) * MB, bh);
        ptx::bulk_commit();
        ptx::bulk_wait<0>();
        // copies still in flight (only after a wait ran out) land before exit
        for (int st = max(0, issued - NSS); st < issued; ++st)
            ptx::mbar_wait_bounded(ptx::smem_addr(&s.full[st % NSS]), (st / NSS) & 1, kDrainNs);
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
            p.bf[(size_t)bh * D + j0] = cb0 + pivot;
            p.bf[(size_t)bh * D + j1] = cb1 + pivot;
        }
    }
}

}  // namespace

bool linear_split_supported(const ttt_desc &d)
{
    return d.io_dtype == TTT_BF16 && d.d == D && d.mini_batch == MB;
}

cudaError_t launch_linear_split(const LinearArgs &a)
{
    const ttt_desc &d = a.desc;
    const int BH = call_rows(d);
    CUtensorMap mq, mk, mv, mz;
    if (!make_bf16_tile_map(&mq, a.Q, d.L, BH, ST) || !make_bf16_tile_map(&mk, a.K, d.L, BH, ST) ||
        !make_bf16_tile_map(&mv, a.V, d.L, BH, ST) || !make_bf16_tile_map(&mz, a.Z, d.L, BH, MB))
        return cudaErrorInvalidValue;
    Params p{d.H, d.L, d.ln_eps, wait_timeout_ns(), withhold_loads(), a.eta, a.W0, a.b0, a.gamma,
             a.beta, a.W_final, a.b_final, a.status, d.init_per_batch};
    p.hoff = head_offset(d);
    const size_t smem = sizeof(Smem) + 1024;
    auto kern = d.residual_ln ? linear_split_kernel<true> : linear_split_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<BH, kThreads, smem, a.stream>>>(mq, mk, mv, mz, p);
    return cudaGetLastError();
}

}  // namespace ttt
