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
// the only sequential dependency is P_n -> G_n -> W_{n+1} -> P_{n+1}.  The
// key-side product of the next mini-batch is re-associated exactly,
//   P_{n+1} = (K_{n+1} W_n + 1 c_n) - ((K_{n+1} K_n^T + 1) diag(eta_n)) G_n,
// so the sequential chain per mini-batch is G_n -> one 16 x 16 x 16 product ->
// G_{n+1}; the d x d update and both d x d products are off that chain.
//
// B300 design.  The scan is latency-bound: 16 tokens of one (batch, head) per
// step, each step waiting on the last.  One CTA per (batch, head), four warps:
//   * 64-token stages of Q, K, V (TMA, 128-byte swizzle) and eta (bulk copy)
//     stream into a 6-deep shared-memory ring; thread 0 refills a slot right after
//     the step barrier that retires it (no separate copy warp);
//   * warps 0-3 each own 16 output features.  W^T lives in registers as fp32
//     warp-MMA accumulators for the whole scan; every contraction is a
//     bf16 m16n8k16 MMA on register fragments, so the recurrence never leaves
//     the register file.  (Measured on B300: a tcgen05 MMA's round trip through
//     tensor memory and an mbarrier takes ~290 cycles and each further MMA ~46
//     cycles of issue; a dependent warp MMA takes ~19 cycles.  On a chain of
//     16-token steps the warp MMA wins.)
//   * each step is one straight-line block on either side of a single named
//     barrier, so the compiler can fill the latency of the LayerNorm chain
//     (shuffle rounds, the barrier, rsqrt) with the off-chain work: the
//     deferred state update, the two d x d products, the 16 x 16 input blocks
//     of the next mini-batch and the previous step's output;
//   * LayerNorm statistics are reduced with a warp reduce-scatter plus one
//     shared-memory exchange; the backward statistics use one pass (sums of z,
//     z^2, g^2 z, g^2 z^2, g b' z, g b' with b' = beta - v + k), all in fp32;
//   * Z tiles are transposed back with stmatrix into a swizzled staging ring
//     and written by TMA stores.
// Inner-learner variants (ai-feeds Modular TTT page: loss and weight decay):
//   * inner-product loss -<f(k), v>: G = -V, or the LayerNorm backward of the upstream
//     -V; the kernel keeps one code path and zeroes the coefficients of the terms the
//     loss does not have (gamma^2 xhat, beta, k);
//   * weight decay lambda (W only, gradient at the mini-batch's start):
//     W_{n+1} = (1 - lambda S_n) W_n - K_n^T diag(eta_n) G_n with S_n the mini-batch's
//     sum of eta, and query token t reads (1 - lambda cum_t) W_n, cum_t the prefix sum
//     of eta up to t.  So the carried W^T is scaled before the deferred update, the
//     output product Y_n and the re-associated key product X_{n+1} are scaled per token
//     around the bias, and the chain is otherwise unchanged (a template switch: the
//     default learner pays none of it).
// Every mbarrier wait is bounded; a wait that runs out sets the library's
// failure flag and the kernel finishes without waiting again.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
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
constexpr int kThreads = 128;
constexpr uint32_t kStageTileBytes = ST * D * 2;   // 8 KB

struct __align__(1024) Smem {
    __nv_bfloat16 q[NSS][ST * D];
    __nv_bfloat16 k[NSS][ST * D];
    __nv_bfloat16 v[NSS][ST * D];
    __nv_bfloat16 z[NZ][MB * D];
    float eta[NSS][ST];
    uint32_t sfrag[3][2][2][32][2];   // [mini-batch % 3][0: chain, 1: output][s half][lane][t n-tile]
    // LayerNorm exchange tables, [parity][token][quantity * 4 + warp].  The token rows are
    // padded (36 and 12 floats) so the 16-byte reads of the four warps' partials are free
    // of bank conflicts and the scattered 4-byte writes are at most 4-way.
    float red[2][MB][36];             // six backward sums (+ 2 spare quantities)
    float zred[2][MB][12];            // output sums: z, z^2
    unsigned long long full[NSS];
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
    int hoff = 0;            // head index of row 0 of this call
    int ip = 0;              // inner-product loss
    float wd = 0.f;          // weight decay lambda (read by the WD instantiation)
};

// Bound of the final wait for copies still in flight (they land in microseconds).
constexpr long long kDrainNs = 1000000000ll;
constexpr long long kDefaultWaitNs = 1000000000ll;

// Slow path of a bounded wait, out of line so the step stays small in the
// instruction cache.  Returns false when the wait ran out (or another one did).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, long long limit, int *abort_flag,
                                       unsigned int *status)
{
    if (*(volatile int *)abort_flag) return false;
    if (ptx::mbar_wait_bounded(bar, parity, limit)) return true;
    *(volatile int *)abort_flag = 1;
    atomicOr(status, kStatusTimeout);
    return false;
}

template <bool LN, bool WD>
__global__ void __launch_bounds__(kThreads, 1)
linear_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmZ,
                    Params p)
{
    extern __shared__ unsigned char smem_raw[];
    // align to 1024 B by offsetting the shared array itself (not through an integer
    // cast), so that plain accesses to the block compile to shared-memory loads/stores
    const uint32_t raw = ptx::smem_addr(smem_raw);
    Smem &s = *reinterpret_cast<Smem *>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, h = (p.hoff + bh) % p.H;
    const int N = p.L / MB;                 // mini-batches
    const int NST = (p.L + ST - 1) / ST;    // stages

    // stage st -> ring slot st % NSS.  There is no copy warp (a waiting copy warp would share
    // a sub-partition with a math warp): thread 0 issues the first stages, and lane 0 of warp
    // 3 (warp 0 already issues the Z stores) refills a slot right after the barrier that
    // retires it.
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
    const int kRefill = 96;
    int issued = min(NSS, nissue);   // stages handed to the copy engine so far
    if (tid == 0) {
        for (int i = 0; i < NSS; ++i) ptx::mbar_init(ptx::smem_addr(&s.full[i]), 1);
        s.abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        for (int st = 0; st < issued; ++st) issue_stage(st);
    }
    __syncthreads();

    // ------------------------------------------------------------------ math warps
    const int g = lane >> 2, c = lane & 3, mrow = lane & 7, mat = lane >> 3;
    const int j0 = warp * 16 + g, j1 = j0 + 8;      // this thread's two features
    bool aborted = false;

    auto wait_stage = [&](int st) {
        if (aborted) return;
        const uint32_t bar = ptx::smem_addr(&s.full[st % NSS]);
        if (ptx::mbar_try_wait(bar, (st / NSS) & 1)) return;
        aborted = !wait_slow(bar, (st / NSS) & 1, p.wait_ns, &s.abort_flag, p.status);
    };
    // shared-memory byte address of row `t` (mini-batch n) / 16-byte chunk of a stage tile.
    // Every caller passes t = 8 k + mrow, so the 128-byte swizzle term (chunk ^ row % 8) is
    // (chunk ^ mrow): the lane part of each address is the same in every step and stays in a
    // register; per step only the tile offset of mini-batch n is added.
    auto tile_addr = [&](const __nv_bfloat16 (*arr)[ST * D], int n, int t, int chunk) -> uint32_t {
        const uint32_t toff = (uint32_t)(((n / TPS) % NSS) * (ST * D * 2) + (n % TPS) * (MB * 128));
        return ptx::smem_addr(arr[0]) + toff + (uint32_t)(t * 128 + ((chunk ^ mrow) << 4));
    };
    auto eta_at = [&](int n, int t) -> float { return s.eta[(n / TPS) % NSS][(n % TPS) * MB + t]; };

    // ---- initial state: W^T rows j0/j1 as fp32 accumulators, c, LN params
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
    float ga0 = 1.f, ga1 = 1.f, be0 = 0.f, be1 = 0.f, C1 = 0.f;
    // LayerNorm pivot: LN(z - p 1) = LN(z) and its backward is unchanged, so with the residual
    // LayerNorm the scan runs on c - p with p = mean(b0), and p is added back to b_final.  The
    // one-pass sums of z and z^2 then see values near zero even when b0 has a large common
    // offset (no cancellation in S2 / D - mu^2).
    float pivot = 0.f;
    if (LN) {
        ga0 = p.gamma[(size_t)h * D + j0];
        ga1 = p.gamma[(size_t)h * D + j1];
        be0 = p.beta[(size_t)h * D + j0];
        be1 = p.beta[(size_t)h * D + j1];
        // sums of gamma^2 and of b0 over all features: this thread's two, the warp, the warps
        float part = ga0 * ga0 + ga1 * ga1, pb = cb0 + cb1;
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
            part += __shfl_xor_sync(0xffffffffu, part, o);
            pb += __shfl_xor_sync(0xffffffffu, pb, o);
        }
        if (lane == 0) {
            s.red[0][0][warp] = part;
            s.red[0][1][warp] = pb;
        }
        ptx::named_bar(1, kMathThreads);
        const float4 w4 = *reinterpret_cast<const float4 *>(s.red[0][0]);
        const float4 p4 = *reinterpret_cast<const float4 *>(s.red[0][1]);
        C1 = p.ip ? 0.f : (w4.x + w4.y) + (w4.z + w4.w);
        pivot = ((p4.x + p4.y) + (p4.z + p4.w)) * (1.f / D);
        cb0 -= pivot;
        cb1 -= pivot;
        ptx::named_bar(1, kMathThreads);
    }
    // LayerNorm backward coefficients: the squared-error loss has gx = gamma (gamma xhat +
    // beta - v + k); the inner-product loss has gx = -gamma v (no gamma^2, beta or k term)
    const float g20 = p.ip ? 0.f : ga0 * ga0, g21 = p.ip ? 0.f : ga1 * ga1;
    const float bx0 = p.ip ? 0.f : be0, bx1 = p.ip ? 0.f : be1;
    const float kf = p.ip ? 0.f : 1.f;   // weight of k in gx, and of P in the plain G

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

    // acc[u][*] = W^T X_n^T + c for a 16-token tile X of mini-batch n (two half-depth
    // accumulator chains per output tile, summed at the end)
    auto product = [&](float (*acc)[4], const __nv_bfloat16 (*arr)[ST * D], int n) {
        uint32_t r[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q)   // matrices: (t-block 0, i-chunk 2q), (t0, 2q+1), (t1, 2q), (t1, 2q+1)
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

    // Input-only 16x16 blocks of mini-batch m, as B fragments (k = source token s,
    // n = target token t):
    //   chain : eta_s (K_{m+1}[t] . K_m[s] + 1)
    //   output: eta_s (Q_m[t] . K_m[s] + 1) [s <= t]
    // warp w: matrix (w >> 1) (0 output, 1 chain), source half (w & 1).  Indices past
    // the sequence are clamped: those blocks are computed but never used.
    auto compute_sfrag = [&](int m) {
        const int which = warp >> 1, half = warp & 1;   // which: 0 output, 1 chain
        const int mm = min(m, N - 1);
        const int na = which ? min(m + 1, N - 1) : mm;
        const __nv_bfloat16(*A)[ST * D] = which ? s.k : s.q;
        uint32_t a[4][4], b[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // A = rows t of the target tile, k = features 16q..16q+15
            // matrices: (t0, chunk 2q), (t1, 2q), (t0, 2q+1), (t1, 2q+1)
            ptx::ldsm_x4(tile_addr(A, na, (mat & 1) * 8 + mrow, 2 * q + (mat >> 1)), a[q]);
            // B = K_m rows s in [8 half, 8 half + 8), k = features: (s, chunk 2q), (s, 2q+1)
            ptx::ldsm_x4(tile_addr(s.k, mm, half * 8 + mrow, 2 * q + (mat & 1)), b[q]);
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, ac2[4] = {0.f, 0.f, 0.f, 0.f};
        ptx::mma_bf16(acc, a[0], b[0][0], b[0][1]);
        ptx::mma_bf16(ac2, a[2], b[2][0], b[2][1]);
        ptx::mma_bf16(acc, a[1], b[1][0], b[1][1]);
        ptx::mma_bf16(ac2, a[3], b[3][0], b[3][1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] += ac2[i];
        // acc: rows t = g (acc0,1), g + 8 (acc2,3); cols s = 8 half + 2c, +1
        const int s0 = half * 8 + 2 * c;
        const float e0 = eta_at(mm, s0), e1 = eta_at(mm, s0 + 1);
        const bool causal = which == 0;   // mask s <= t on the output block
        const float v0 = (causal && s0 > g) ? 0.f : e0 * (acc[0] + 1.f);
        const float v1 = (causal && s0 + 1 > g) ? 0.f : e1 * (acc[1] + 1.f);
        const float v2 = (causal && s0 > g + 8) ? 0.f : e0 * (acc[2] + 1.f);
        const float v3 = (causal && s0 + 1 > g + 8) ? 0.f : e1 * (acc[3] + 1.f);
        uint32_t *dst = s.sfrag[m % 3][which ? 0 : 1][half][lane];
        *reinterpret_cast<uint2 *>(dst) = make_uint2(ptx::pack_bf16(v0, v1), ptx::pack_bf16(v2, v3));
    };
    auto read_sfrag = [&](int m, int which, uint32_t (*b)[2]) {   // b[u][half]
        const uint2 f0 = *reinterpret_cast<const uint2 *>(s.sfrag[m % 3][which][0][lane]);
        const uint2 f1 = *reinterpret_cast<const uint2 *>(s.sfrag[m % 3][which][1][lane]);
        b[0][0] = f0.x; b[1][0] = f0.y;
        b[0][1] = f1.x; b[1][1] = f1.y;
    };

    // reduce-scatter of 8 per-token values (4 tokens x 2 quantities) over the 8 lanes
    // sharing c; the lane keeps token t_own (below), quantity g & 1
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
    // token of this lane after a reduce-scatter: tk = g / 2 -> t = 8 (tk / 2) + 2c + (tk % 2)
    const int tk = g >> 1, qh = g & 1;
    const int t_own = 8 * (tk >> 1) + 2 * c + (tk & 1);

    // per-token output sums of Zbar (for the output LayerNorm), scattered into zred
    auto zbar_stats = [&](const float (*zb)[4], int par) {
        float zs[8];
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) {
            const int u = tq >> 1, e = tq & 1;
            const float z0 = zb[u][e], z1 = zb[u][2 + e];
            zs[tq * 2 + 0] = z0 + z1;
            zs[tq * 2 + 1] = fmaf(z0, z0, z1 * z1);
        }
        s.zred[par][t_own][4 * qh + warp] = rs8(zs);
    };

    // Z_m = Q_m + LN(Zbar_m) (or Zbar_m) -> bf16 staging tile m % NZ
    auto finish_z = [&](const float (*zb)[4], const float (*qv)[4], int m, int par) {
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
                z[u][e] = qv[u][e] + fmaf(ga0 * (zb[u][e] - m_t), r_t, be0);
                z[u][2 + e] = qv[u][2 + e] + fmaf(ga1 * (zb[u][2 + e] - m_t), r_t, be1);
            }
        } else {
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) z[u][i] = zb[u][i];
        }
        uint32_t r[4];
        r[0] = ptx::pack_bf16(z[0][0], z[0][1]);
        r[1] = ptx::pack_bf16(z[0][2], z[0][3]);
        r[2] = ptx::pack_bf16(z[1][0], z[1][1]);
        r[3] = ptx::pack_bf16(z[1][2], z[1][3]);
        // matrices (j-block, t-block): (0,0), (1,0), (0,1), (1,1); stored rows = tokens
        const uint32_t zaddr = ptx::smem_addr(s.z[m % NZ]);
        ptx::stsm_x4_t(zaddr + ptx::sw128((mat >> 1) * 8 + mrow, warp * 2 + (mat & 1)), r);
        ptx::fence_proxy_async();
    };

    // W^T += (-eta G_m)^T K_m, as 8 independent accumulator tiles
    auto update_w = [&](const uint32_t *nge, int m) {
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
            // matrices (s-block, i-chunk): (0, 2pp), (1, 2pp), (0, 2pp+1), (1, 2pp+1)
            uint32_t r[4];
            ptx::ldsm_x4_t(tile_addr(s.k, m, (mat & 1) * 8 + mrow, 2 * pp + (mat >> 1)), r);
            ptx::mma_bf16(wt[2 * pp], nge, r[0], r[1]);
            ptx::mma_bf16(wt[2 * pp + 1], nge, r[2], r[3]);
        }
    };

    // ---- prologue: P_0 = K_0 W_0 + c_0, input blocks of mini-batch 0
    wait_stage(0);
    if (N > TPS) wait_stage(1);
    pack_w();
    float pacc[2][4];
    product(pacc, s.k, 0);
    compute_sfrag(0);
    ptx::named_bar(1, kMathThreads);

    // carried between steps: the previous step's -eta G (deferred W update), its output
    float zprev[2][4] = {}, qprev[2][4] = {};
    uint32_t ngep[4] = {0u, 0u, 0u, 0u};
    float dprev = 1.f;   // weight decay: 1 - lambda S_{n-1}, the factor of the deferred update

    // weight decay: scale the carried W^T by 1 - lambda S before the deferred update
    auto decay_w = [&](float f) {
#pragma unroll
        for (int pt = 0; pt < 8; ++pt)
#pragma unroll
            for (int i = 0; i < 4; ++i) wt[pt][i] *= f;
    };

    for (int n = 0; n < N; ++n) {
        const int par = n & 1;
        // the input blocks of mini-batch n + 1 read K_{n+2}: its stage must have landed
        if ((n + 2) % TPS == 0 && n + 2 < N) wait_stage((n + 2) / TPS);

        // ======== before the barrier ========
        // input blocks of the next mini-batch (independent of the state)
        if (LN) compute_sfrag(n + 1);
        // deferred update with G_{n-1} (zero fragments at n = 0): W_n, then its bf16 copy
        if (WD) decay_w(dprev);
        update_w(ngep, max(n - 1, 0));
        pack_w();
        // weight decay: per-token factors 1 - lambda cum_t for this lane's tokens 8u + 2c + e
        // (prefix sums of eta within the mini-batch by a scan over the 4 lanes sharing g)
        float fq[2][2] = {{1.f, 1.f}, {1.f, 1.f}}, dn = 1.f;
        if (WD) {
            const float a0 = eta_at(n, 2 * c), a1 = eta_at(n, 2 * c + 1);
            const float b0 = eta_at(n, 2 * c + 8), b1 = eta_at(n, 2 * c + 9);
            float ia = a0 + a1, ib = b0 + b1;
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                const float ta = __shfl_up_sync(0xffffffffu, ia, o, 4);
                const float tb = __shfl_up_sync(0xffffffffu, ib, o, 4);
                if (c >= o) {
                    ia += ta;
                    ib += tb;
                }
            }
            const float ta = __shfl_sync(0xffffffffu, ia, 3, 4);   // sum over tokens 0..7
            const float tb = __shfl_sync(0xffffffffu, ib, 3, 4);
            fq[0][0] = 1.f - p.wd * (ia - a1);
            fq[0][1] = 1.f - p.wd * ia;
            fq[1][0] = 1.f - p.wd * (ta + ib - b1);
            fq[1][1] = 1.f - p.wd * (ta + ib);
            dn = 1.f - p.wd * (ta + tb);
        }
        // products from W_n: output Y_n = W_n^T Q_n^T + c_n, and the key product of the
        // next mini-batch (clamped at the end: unused)
        float yacc[2][4], xacc[2][4];
        product(yacc, s.q, n);
        // with LayerNorm the pre-barrier shuffle rounds hide this product; without it the
        // step is short on both sides and the product balances the post-barrier half
        if (LN) product(xacc, s.k, min(n + 1, N - 1));
        float vt[2][4], qt[2][4];
        load_T(vt, s.v, n);
        load_T(qt, s.q, n);
        float gb[2][4];
        if (LN) {
            float kt[2][4];
            load_T(kt, s.k, n);
            // b'_j = beta_j - (v - k); gb = gamma * b'
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                gb[u][0] = ga0 * fmaf(kt[u][0], kf, bx0 - vt[u][0]);
                gb[u][1] = ga0 * fmaf(kt[u][1], kf, bx0 - vt[u][1]);
                gb[u][2] = ga1 * fmaf(kt[u][2], kf, bx1 - vt[u][2]);
                gb[u][3] = ga1 * fmaf(kt[u][3], kf, bx1 - vt[u][3]);
            }
            // per-token partial sums over this thread's two features
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
            // lane holds token t_own, quantities 3 qh + 0..2
#pragma unroll
            for (int i = 0; i < 3; ++i) s.red[par][t_own][4 * (3 * qh + i) + warp] = a3[i];
            // output statistics of the previous step ride on the same barrier
            zbar_stats(zprev, par);
        }
        if (!LN) compute_sfrag(n + 1);
        if (warp == 0 && lane == 0) ptx::bulk_wait_read<NZ - 2>();
        ptx::named_bar(1, kMathThreads);

        // ======== after the barrier ========
        if (!LN) product(xacc, s.k, min(n + 1, N - 1));
        // G_n
        float gmat[2][4];
        if (LN) {
            // totals for (t_own, 3 qh + i), then the partner lane supplies the other three
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
                for (int i = 0; i < 4; ++i) gmat[u][i] = fmaf(pacc[u][i], kf, -vt[u][i]);
        }

        // -G and -eta G as A fragments (rows = features, k = tokens)
        const int s0 = 2 * c;
        const float e00 = eta_at(n, s0), e01 = eta_at(n, s0 + 1);
        const float e10 = eta_at(n, s0 + 8), e11 = eta_at(n, s0 + 9);
        uint32_t ng[4];
        ng[0] = ptx::pack_bf16(-gmat[0][0], -gmat[0][1]);
        ng[1] = ptx::pack_bf16(-gmat[0][2], -gmat[0][3]);
        ng[2] = ptx::pack_bf16(-gmat[1][0], -gmat[1][1]);
        ng[3] = ptx::pack_bf16(-gmat[1][2], -gmat[1][3]);
        // chain: P_{n+1} = X_{n+1} - G_n^T M^T; with weight decay
        // X_{n+1} = (1 - lambda S_n) K_{n+1} W_n + c_n
        uint32_t bf[2][2];
        read_sfrag(n, 0, bf);
        if (WD) {
            const float l0 = (1.f - dn) * cb0, l1 = (1.f - dn) * cb1;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                xacc[u][0] = fmaf(dn, xacc[u][0], l0);
                xacc[u][1] = fmaf(dn, xacc[u][1], l0);
                xacc[u][2] = fmaf(dn, xacc[u][2], l1);
                xacc[u][3] = fmaf(dn, xacc[u][3], l1);
                // Y_n: token t reads (1 - lambda cum_t) W_n
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float f = fq[u][e];
                    yacc[u][e] = fmaf(f, yacc[u][e], (1.f - f) * cb0);
                    yacc[u][2 + e] = fmaf(f, yacc[u][2 + e], (1.f - f) * cb1);
                }
            }
            dprev = dn;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
#pragma unroll
            for (int i = 0; i < 4; ++i) pacc[u][i] = xacc[u][i];
            ptx::mma_bf16(pacc[u], ng, bf[u][0], bf[u][1]);
        }
        // output: Zbar_n = Y_n - G_n^T B^T
        read_sfrag(n, 1, bf);
#pragma unroll
        for (int u = 0; u < 2; ++u) ptx::mma_bf16(yacc[u], ng, bf[u][0], bf[u][1]);
        // deferred W update operand, and c -= eta^T G now
        ngep[0] = ptx::pack_bf16(-e00 * gmat[0][0], -e01 * gmat[0][1]);
        ngep[1] = ptx::pack_bf16(-e00 * gmat[0][2], -e01 * gmat[0][3]);
        ngep[2] = ptx::pack_bf16(-e10 * gmat[1][0], -e11 * gmat[1][1]);
        ngep[3] = ptx::pack_bf16(-e10 * gmat[1][2], -e11 * gmat[1][3]);
        {
            float d0 = e00 * gmat[0][0] + e01 * gmat[0][1] + e10 * gmat[1][0] + e11 * gmat[1][1];
            float d1 = e00 * gmat[0][2] + e01 * gmat[0][3] + e10 * gmat[1][2] + e11 * gmat[1][3];
            d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
            d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
            cb0 -= d0;
            cb1 -= d1;
        }
        // the previous output (its statistics crossed this barrier); at n = 0 this
        // writes a tile that is overwritten before it is ever stored
        finish_z(zprev, qprev, n + NZ - 1, par);
        if (warp == 0 && lane == 0) {
            // Z_{n-2} was finished before this step's barrier
            if (n >= 2) {
                ptx::tma_store_3d(&tmZ, ptx::smem_addr(s.z[(n - 2) % NZ]), 0, (n - 2) * MB, bh);
                ptx::bulk_commit();
            }
        }
        if (tid == kRefill && n >= TPS && n % TPS == 0 && n / TPS - 1 + NSS < nissue && !aborted) {
            // the stage holding n - 1 is no longer read (its last reader, the update with
            // G_{n-1}, ran before this step's barrier): refill its slot
            ptx::fence_proxy_async();
            issue_stage(n / TPS - 1 + NSS);
            issued = n / TPS + NSS;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                zprev[u][i] = yacc[u][i];
                qprev[u][i] = qt[u][i];
            }
    }

    // ---- tail: last update, last output, final stores, final state
    if (WD) decay_w(dprev);
    update_w(ngep, N - 1);
    {
        const int par = N & 1;
        if (LN) zbar_stats(zprev, par);
        if (warp == 0 && lane == 0) ptx::bulk_wait_read<NZ - 2>();
        ptx::named_bar(1, kMathThreads);
        finish_z(zprev, qprev, N - 1, par);
        ptx::named_bar(1, kMathThreads);
        if (warp == 0 && lane == 0) {
            for (int n = max(0, N - 2); n < N; ++n) {
                ptx::tma_store_3d(&tmZ, ptx::smem_addr(s.z[n % NZ]), 0, n * MB, bh);
                ptx::bulk_commit();
            }
            ptx::bulk_wait<0>();
        }
    }
    if (tid == kRefill)   // copies still in flight (only after a wait ran out) land before exit
        for (int st = max(0, issued - NSS); st < issued; ++st)
            ptx::mbar_wait_bounded(ptx::smem_addr(&s.full[st % NSS]), (st / NSS) & 1, kDrainNs);
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

// test hooks: process-wide, set by any host thread and read when a call launches
std::atomic<long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_withhold_loads{0};

}  // namespace

// [rows][cols] bf16 row-major as a 2-D tensor; boxes of box_rows x 64 columns, 128-byte swizzle.
bool make_bf16_2d_map(CUtensorMap *m, const void *base, unsigned long long rows, unsigned long long cols,
                      unsigned box_rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// [BH][L][64] bf16 viewed as a 3-D tensor; boxes of `rows` tokens, 128-byte swizzle.
bool make_bf16_tile_map(CUtensorMap *m, const void *base, int L, int BH, int rows)
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

void set_wait_timeout_ns(long long ns) { g_wait_ns.store(ns > 0 ? ns : kDefaultWaitNs, std::memory_order_relaxed); }
void set_withhold_loads(int on) { g_withhold_loads.store(on != 0, std::memory_order_relaxed); }
long long wait_timeout_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int withhold_loads() { return g_withhold_loads.load(std::memory_order_relaxed); }

bool linear_tc_supported(const ttt_desc &d)
{
    return d.io_dtype == TTT_BF16 && d.d == D && d.mini_batch == MB;
}

cudaError_t launch_linear_tc(const LinearArgs &a)
{
    const ttt_desc &d = a.desc;
    const int BH = call_rows(d);
    CUtensorMap mq, mk, mv, mz;
    if (!make_bf16_tile_map(&mq, a.Q, d.L, BH, ST) || !make_bf16_tile_map(&mk, a.K, d.L, BH, ST) ||
        !make_bf16_tile_map(&mv, a.V, d.L, BH, ST) || !make_bf16_tile_map(&mz, a.Z, d.L, BH, MB))
        return cudaErrorInvalidValue;
    Params p{d.H, d.L, d.residual_ln, d.ln_eps, wait_timeout_ns(), withhold_loads(), a.eta, a.W0, a.b0, a.gamma, a.beta,
             a.W_final, a.b_final, a.status, d.init_per_batch};
    p.hoff = head_offset(d);
    p.ip = d.loss == TTT_LOSS_INNER_PRODUCT;
    p.wd = d.weight_decay;
    const size_t smem = sizeof(Smem) + 1024;
    const bool wd = d.weight_decay != 0.f;
    auto kern = d.residual_ln ? (wd ? linear_fused_kernel<true, true> : linear_fused_kernel<true, false>)
                              : (wd ? linear_fused_kernel<false, true> : linear_fused_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<BH, kThreads, smem, a.stream>>>(mq, mk, mv, mz, p);
    return cudaGetLastError();
}

}  // namespace ttt
