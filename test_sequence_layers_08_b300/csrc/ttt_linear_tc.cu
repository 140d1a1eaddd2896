// ttt_linear_tc.cu -- fused TTT-Linear forward for bf16 I/O, d = 64, b = 16.
//
// The method (damodev.csdn.net TTT article, sections 3.1 and 4.1-4.2; residual
// LayerNorm of the lryc.cn TTT article, section 2.1): per (batch, head) the
// fast weights (W, c) are updated once per mini-batch of 16 tokens, every
// token's gradient taken at the mini-batch's starting weights, and each output
// read with the weights after its own token's update:
//   P_n = K_n W_n + 1 c_n                        (key-side forward, 16 x 64)
//   G_n = P_n - V_n  or  LNbwd(P_n; V_n - K_n)   (per-token gradient)
//   W_{n+1} = W_n - K_n^T diag(eta_n) G_n,  c_{n+1} = c_n - eta_n^T G_n
//   Z_n = f_out(Q_n W_n + 1 c_n - tril(Q_n K_n^T + 1) diag(eta_n) G_n).
//
// The only sequential dependency is G_n -> P_{n+1}.  It is shortened with an
// exact four-step lookahead: with C_{t,l} = K_t K_l^T + 1,
//   P_t = (K_t W_{t-4} + 1 c_{t-4}) - sum_{l=t-4}^{t-1} C_{t,l} diag(eta_l) G_l.
// The product with W_{t-4} and the corrections from G_{t-4}, G_{t-3} run on the
// tcgen05 tensor cores well ahead of time; only the two newest corrections
// (16 x 16 x 64 each) and the LayerNorm backward sit on the chain, on warp MMAs.
//
// B300 design.  One CTA (14 warps) per (batch, head):
//   * warp 12 streams 64-token stages of K, Q, V (TMA, 128-byte swizzle) and
//     eta (bulk copy) into a 5-deep ring;
//   * warp 13 issues every tcgen05 MMA: per stage the Gram block
//     [K_s; Q_s] [K_{s-1}; K_s]^T; per step the state update
//     W~^T -= (eta G)^T [K | 1] into one of two TMEM accumulators (W~ = [W; c],
//     alternating so that reading one never stalls the next update), the
//     products K_{n+4} W~_n and Q_n W~_n (bias folded in through a column of
//     ones), the output correction and the lookahead corrections;
//   * warps 0-3 ("chain") each own 16 output features: they finish P_n, compute
//     G_n with the LayerNorm statistics reduced in fp32 (warp shuffles and one
//     shared-memory exchange, and publish (eta G_n)^T for the tensor cores;
//   * warps 4-7 convert the fp32 TMEM state into the bf16 operand tile the
//     products read, and cut the Gram blocks into masked bf16 operands;
//   * warps 8-11 (one per mini-batch of a stage) finish the outputs: residual
//     LayerNorm, bf16 conversion, TMA store.
// TMEM (512 columns): two W~^T accumulators (2 x 80), six lookahead
// accumulators (6 x 16), two output accumulators (2 x 64), one Gram (128).
// Every mbarrier wait is bounded; a wait that runs out sets the library's
// failure flag, and from then on no role waits again, so the kernel finishes.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int D = 64;          // head dim
constexpr int MB = 16;         // mini-batch
constexpr int ST = 64;         // tokens per pipeline stage
constexpr int TPS = ST / MB;   // mini-batches per stage
constexpr int NSS = 5;         // stage ring depth
constexpr int XR = 6;          // lookahead accumulators
constexpr int GR = 4;          // (eta G)^T tiles
constexpr int PS = 3;          // prepared-operand slots (one per stage)
constexpr int YR = 2;          // output accumulators
constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;
constexpr int kAux0 = 4, kEpi0 = 8, kProd = 12, kIssue = 13;

constexpr uint32_t TM_W = 0;     // 2 x 80 columns: W^T (64) and the bias tile (column 64)
constexpr uint32_t TM_X = 160;   // XR x 16
constexpr uint32_t TM_Y = 256;   // YR x 64
constexpr uint32_t TM_G = 384;   // 128
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t kTileBytes = ST * D * 2;   // 8 KB

struct __align__(1024) Smem {
    __nv_bfloat16 stage[NSS][3][ST * D];     // [slot][0 K, 1 Q, 2 V], 128-byte swizzled rows
    __nv_bfloat16 wt[2][D * D];              // bf16 W^T [j][i], 128-byte swizzle
    __nv_bfloat16 zst[4][MB * D];            // Z staging, one per epilogue warp
    __nv_bfloat16 cb[PS][TPS][2][MB * MB];   // lookahead B tiles [t][s]: [0] C_{t,t-4}, [1] C_{t,t-3}
    __nv_bfloat16 bout[PS][ST * MB];         // output-correction A tiles [t'][s]
    __nv_bfloat16 gt[GR][D * MB];            // (eta G)^T [j][s]
    __nv_bfloat16 ct[2][D * MB];             // bias tile [j][16], column 0 = c_j
    __nv_bfloat16 onesA[ST * MB];            // [t'][16], column 0 = 1
    __nv_bfloat16 onesB[MB * MB];            // [t][16], column 0 = 1
    __nv_bfloat16 onesR[MB * MB];            // [n][16], row 0 = 1
    uint32_t cfrag[PS][TPS][2][32][4];       // chain A fragments: [0] -C_{t,t-2}, [1] -C_{t,t-1}
    float xtr[4][MB * 20];                   // chain transposes
    float stats[3][MB][8];                   // per-token LayerNorm sums
    float eta[NSS][ST];
    unsigned long long full[NSS], empty[NSS];
    unsigned long long gram_full, prep_full[PS], prep_free[PS];
    unsigned long long wbuf_full[2], wbuf_free[2], wupd_full[2];
    unsigned long long x_full[XR];
    unsigned long long g_full[GR], g_free[GR];
    unsigned long long z_full[TPS], y_free[YR];   // z_full: one per epilogue warp
    unsigned long long fin;
    uint32_t tmem;
    int abort_flag;
};

struct Params {
    int H, L, N, NST, init_per_batch;
    float eps;
    long long wait_ns;
    int withhold_loads;
    const float *eta, *W0, *b0, *gamma, *beta;
    float *Wf, *bf;
    unsigned int *status;
};

static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory budget");

constexpr long long kDrainNs = 1000000000ll;
constexpr long long kDefaultWaitNs = 1000000000ll;

// Bounded waits sharing one abort flag: once any wait has run out, every
// later wait returns at once and the roles run to the end without blocking.
// The first wait to run out records, in the failure flag, which barrier of
// which role gave up at which step (bit 0: timeout; bits 8-19: step mod 4096;
// bits 20-27: barrier index in the shared-memory block; bits 28-31: role).
struct Waiter {
    int *abort_flag;
    unsigned int *status;
    long long ns;
    const unsigned long long *bar0;
    unsigned int role;
    __device__ __forceinline__ bool operator()(unsigned long long *bar, uint32_t parity, int step = 0) const
    {
        if (*(volatile int *)abort_flag) return false;
        const uint32_t a = ptx::smem_addr(bar);
        if (ptx::mbar_try_wait(a, parity)) return true;
        const unsigned long long t0 = ptx::globaltimer_ns();
        for (;;) {
            for (int i = 0; i < 32; ++i)
                if (ptx::mbar_try_wait(a, parity)) return true;
            if (*(volatile int *)abort_flag) return false;
            if ((long long)(ptx::globaltimer_ns() - t0) > ns) break;
        }
        if (atomicExch(abort_flag, 1) == 0) {
            const unsigned int idx = (unsigned int)(bar - bar0) & 0xffu;
            atomicCAS(status, 0u, kStatusTimeout | ((unsigned int)(step & 0xfff) << 8) | (idx << 20) |
                                      (role << 28));
            atomicOr(status, kStatusTimeout);
        }
        return false;
    }
};

__device__ __forceinline__ uint32_t bar_addr(unsigned long long *b) { return ptx::smem_addr(b); }

// ---------------------------------------------------------------------------
// roles
// ---------------------------------------------------------------------------

__device__ __forceinline__ void producer(Smem &s, const Params &p, const CUtensorMap *tmK,
                                         const CUtensorMap *tmQ, const CUtensorMap *tmV, int bh,
                                         const Waiter &wait)
{
    ptx::prefetch_tmap(tmK);
    ptx::prefetch_tmap(tmQ);
    ptx::prefetch_tmap(tmV);
    const float *eta_bh = p.eta + (size_t)bh * p.L;
    int issued = 0;
    for (int st = 0; st < (p.withhold_loads ? 0 : p.NST); ++st) {
        const int b = st % NSS;
        if (st >= NSS && !wait(&s.empty[b], ((st / NSS) - 1) & 1, st)) break;
        const int ntok = min(ST, p.L - st * ST);
        const uint32_t fb = bar_addr(&s.full[b]);
        ptx::mbar_arrive_expect_tx(fb, 3 * kTileBytes + ntok * 4);
        ptx::tma_load_3d(ptx::smem_addr(s.stage[b][0]), tmK, fb, 0, st * ST, bh);
        ptx::tma_load_3d(ptx::smem_addr(s.stage[b][1]), tmQ, fb, 0, st * ST, bh);
        ptx::tma_load_3d(ptx::smem_addr(s.stage[b][2]), tmV, fb, 0, st * ST, bh);
        ptx::bulk_load(ptx::smem_addr(s.eta[b]), eta_bh + st * ST, ntok * 4, fb);
        issued = st + 1;
    }
    // every copy issued must land before the CTA may exit
    for (int st = max(0, issued - NSS); st < issued; ++st)
        ptx::mbar_wait_bounded(bar_addr(&s.full[st % NSS]), (st / NSS) & 1, kDrainNs);
}

__device__ __forceinline__ void issuer(Smem &s, const Params &p, uint32_t tm, const Waiter &wait)
{
    const int N = p.N, NST = p.NST;
    constexpr uint32_t idG = ptx::idesc_bf16(128, 64, false, false, false);
    constexpr uint32_t idX = ptx::idesc_bf16(64, 16, false, false, false);
    constexpr uint32_t idY = ptx::idesc_bf16(64, 64, false, false, false);
    constexpr uint32_t idW = ptx::idesc_bf16(64, 64, false, true, true);
    constexpr uint32_t idC = ptx::idesc_bf16(64, 16, false, false, true);
    constexpr uint32_t idO = ptx::idesc_bf16(64, 64, false, false, true);
    constexpr uint32_t idK = ptx::idesc_bf16(64, 16, false, false, true);
    const uint32_t onesA = ptx::smem_addr(s.onesA), onesB = ptx::smem_addr(s.onesB);
    const uint32_t onesR = ptx::smem_addr(s.onesR);

    auto ktile = [&](int st) { return ptx::smem_addr(s.stage[st % NSS][0]); };
    auto qtile = [&](int st) { return ptx::smem_addr(s.stage[st % NSS][1]); };
    auto gram = [&](int st) {
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = ptx::sdesc_sw128(ktile(st) + 32 * kk);   // [K_st; Q_st]: 128 rows
            ptx::tc_mma(tm + TM_G + 64, a, ptx::sdesc_sw128(ktile(st) + 32 * kk), idG, kk > 0);
            if (st > 0)
                ptx::tc_mma(tm + TM_G, a, ptx::sdesc_sw128(ktile(st - 1) + 32 * kk), idG, kk > 0);
        }
        ptx::tc_commit(bar_addr(&s.gram_full));
    };
    // X''_t = W~_wb^T [K_t | 1]^T  (features x tokens)
    auto product_x = [&](int t, int wb) {
        const uint32_t d = tm + TM_X + 16 * (t % XR);
        const uint32_t kb = ktile(t / TPS) + (t % TPS) * MB * 128;
        const uint32_t w = ptx::smem_addr(s.wt[wb]);
        for (int kk = 0; kk < 4; ++kk)
            ptx::tc_mma(d, ptx::sdesc_sw128(w + 32 * kk), ptx::sdesc_sw128(kb + 32 * kk), idX, kk > 0);
        ptx::tc_mma(d, ptx::sdesc_sw32(ptx::smem_addr(s.ct[wb])), ptx::sdesc_sw32(onesB), idX, 1);
    };

    // ---- prologue: Gram of stage 0, lookahead products of targets 0..3 from W_0
    if (wait(&s.full[0], 0)) ptx::tc_fence_after();
    gram(0);
    if (wait(&s.wbuf_full[0], 0)) ptx::tc_fence_after();
    for (int t = 0; t < min(4, N); ++t) product_x(t, 0);
    for (int t = 0; t < min(3, N); ++t) ptx::tc_commit(bar_addr(&s.x_full[t % XR]));
    wait(&s.prep_full[0], 0);
    if (NST > 1) {
        if (wait(&s.full[1 % NSS], 0)) ptx::tc_fence_after();
        gram(1);
    }

    for (int n = 0; n < N; ++n) {
        const int st = n / TPS, m = n % TPS;
        // ---- (A1) as soon as G_n is published: the state update (critical for the
        // products four steps ahead) and the last tensor-core correction of target n + 3
        if (wait(&s.g_full[n % GR], (n / GR) & 1, n)) ptx::tc_fence_after();
        const uint32_t g_n = ptx::smem_addr(s.gt[n % GR]);
        {
            // W~_{n+1} = W~_{n-1} - (eta G)^T [K | 1] for l = n-1, n (accumulator (n+1) % 2);
            // the converter finished reading W~_{n-1} before W~_n was released to step n's products
            const uint32_t d = tm + TM_W + 80 * ((n + 1) & 1);
            for (int l = max(0, n - 1); l <= n; ++l) {
                const uint32_t gl = ptx::smem_addr(s.gt[l % GR]);
                const uint32_t kb = ktile(l / TPS) + (l % TPS) * MB * 128;
                ptx::tc_mma(d, ptx::sdesc_sw32(gl), ptx::sdesc_sw128_mn(kb), idW, 1);
                ptx::tc_mma(d + 64, ptx::sdesc_sw32(gl), ptx::sdesc_sw32(onesR), idC, 1);
            }
            ptx::tc_commit(bar_addr(&s.wupd_full[(n + 1) & 1]));
        }
        if (n + 3 < N) {
            const int t = n + 3;
            ptx::tc_mma(tm + TM_X + 16 * (t % XR), ptx::sdesc_sw32(g_n),
                        ptx::sdesc_sw32(ptx::smem_addr(s.cb[(t / TPS) % PS][t % TPS][1])), idK, 1);
            ptx::tc_commit(bar_addr(&s.x_full[t % XR]));
        }
        // ---- (B) products of W~_n: the output of step n and the lookahead of target n + 4
        if (m == 0) {
            if (st + 1 < NST) wait(&s.prep_full[(st + 1) % PS], ((st + 1) / PS) & 1, n);
            if (st + 2 < NST) {
                if (wait(&s.full[(st + 2) % NSS], ((st + 2) / NSS) & 1, n)) ptx::tc_fence_after();
                gram(st + 2);
            }
        }
        const int wb = n & 1;
        if (n > 0) wait(&s.wbuf_full[wb], (n >> 1) & 1, n);
        if (n >= YR) wait(&s.y_free[n % YR], ((n - YR) / YR) & 1, n);
        ptx::tc_fence_after();
        {
            // Y_n = [Q_stage | 1] W~_n  (stage tokens x features; rows of mini-batch m are valid)
            const uint32_t d = tm + TM_Y + 64 * (n % YR);
            const uint32_t w = ptx::smem_addr(s.wt[wb]);
            for (int kk = 0; kk < 4; ++kk)
                ptx::tc_mma(d, ptx::sdesc_sw128(qtile(st) + 32 * kk), ptx::sdesc_sw128(w + 32 * kk), idY,
                            kk > 0);
            ptx::tc_mma(d, ptx::sdesc_sw32(onesA), ptx::sdesc_sw32(ptx::smem_addr(s.ct[wb])), idY, 1);
        }
        if (n + 4 < N) product_x(n + 4, wb);
        ptx::tc_commit(bar_addr(&s.wbuf_free[wb]));
        // ---- (A2) the terms of G_n that need this step's products: output correction
        // Y_n -= tril(Q K^T + 1) (eta G), and the first correction of target n + 4
        ptx::tc_mma(tm + TM_Y + 64 * (n % YR), ptx::sdesc_sw32(ptx::smem_addr(s.bout[st % PS])),
                    ptx::sdesc_sw32(g_n), idO, 1);
        ptx::tc_commit(bar_addr(&s.z_full[n % TPS]));
        if (n + 4 < N) {
            const int t = n + 4;
            ptx::tc_mma(tm + TM_X + 16 * (t % XR), ptx::sdesc_sw32(g_n),
                        ptx::sdesc_sw32(ptx::smem_addr(s.cb[(t / TPS) % PS][t % TPS][0])), idK, 1);
        }
        if (n >= 1) ptx::tc_commit(bar_addr(&s.g_free[(n - 1) % GR]));
        if (m == TPS - 1 || n == N - 1) ptx::tc_commit(bar_addr(&s.prep_free[st % PS]));
        if (n >= 1 && (n - 1) % TPS == TPS - 1) ptx::tc_commit(bar_addr(&s.empty[((n - 1) / TPS) % NSS]));
        if (n == N - 1) ptx::tc_commit(bar_addr(&s.empty[st % NSS]));
    }
    // every MMA must be complete before the tensor memory is released
    ptx::tc_commit(bar_addr(&s.fin));
    ptx::mbar_wait_bounded(bar_addr(&s.fin), 0, kDrainNs);
}

// Converter + operand preparation (warps 4-7; quarter q of the TMEM lanes).
template <bool LN>
__device__ __forceinline__ void aux(Smem &s, const Params &p, uint32_t tm, int q, int bh,
                                    const Waiter &wait)
{
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int N = p.N;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;

    // W^T fragment registers (rows 16q + g (+8), columns 8k + 2c (+1)) -> bf16 tile
    auto write_wtile = [&](int buf, const float *w) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            pk[2 * k] = ptx::pack_bf16(w[4 * k], w[4 * k + 1]);
            pk[2 * k + 1] = ptx::pack_bf16(w[4 * k + 2], w[4 * k + 3]);
        }
        const uint32_t base = ptx::smem_addr(s.wt[buf]);
        const int sel = lane >> 3, r = lane & 7;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = 2 * i + (sel >> 1), row = 16 * q + 8 * (sel & 1) + r;
            ptx::stsm_x4(base + ptx::sw128(row, k), pk + 4 * i);
        }
    };
    auto write_bias = [&](int buf, float c_lo, float c_hi) {
        if (c == 0) {
            __nv_bfloat16 *ct = s.ct[buf];
            const int r0 = 16 * q + g, r1 = r0 + 8;
            *reinterpret_cast<__nv_bfloat16 *>(reinterpret_cast<unsigned char *>(ct) + ptx::sw32(r0, 0)) =
                __float2bfloat16_rn(c_lo);
            *reinterpret_cast<__nv_bfloat16 *>(reinterpret_cast<unsigned char *>(ct) + ptx::sw32(r1, 0)) =
                __float2bfloat16_rn(c_hi);
        }
    };

    // ---- initial state into both TMEM accumulators and the first bf16 tile
    {
        const size_t init = p.init_per_batch ? (size_t)bh : (size_t)(bh % p.H);
        const float *W0 = p.W0 + init * D * D;
        const float *b0 = p.b0 + init * D;
        float w[32];
        const int j0 = 16 * q + g, j1 = j0 + 8;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = 8 * k + 2 * c;
            w[4 * k] = W0[i * D + j0];
            w[4 * k + 1] = W0[(i + 1) * D + j0];
            w[4 * k + 2] = W0[i * D + j1];
            w[4 * k + 3] = W0[(i + 1) * D + j1];
        }
        const float c_lo = b0[j0], c_hi = b0[j1];
        uint32_t wr[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) wr[i] = __float_as_uint(w[i]);
        uint32_t cr[4] = {c == 0 ? __float_as_uint(c_lo) : 0u, 0u, c == 0 ? __float_as_uint(c_hi) : 0u, 0u};
        for (int b = 0; b < 2; ++b) {
            ptx::tc_st16_x8(tm + TM_W + 80 * b + lane_base, wr);
            ptx::tc_st16_x1(tm + TM_W + 80 * b + 64 + lane_base, cr);
        }
        ptx::tc_wait_st();
        write_wtile(0, w);
        write_bias(0, c_lo, c_hi);
        ptx::fence_proxy_async();
        __syncwarp();
        ptx::tc_fence_before();
        if (lane == 0) ptx::mbar_arrive(bar_addr(&s.wbuf_full[0]));
    }

    // ---- operand preparation for target t (blocks whose rows live in this quarter)
    auto prep = [&](int t) {
        const int st = t / TPS, mt = t % TPS, ps = st % PS;
        if (mt == 0) {
            if (st >= PS) wait(&s.prep_free[ps], ((st / PS) - 1) & 1, t);
            if (wait(&s.gram_full, st & 1, t)) ptx::tc_fence_after();
        }
        if (q == (mt >> 1)) {
            // K_t rows: C_{t,l} = K_t K_l^T + 1 for l = t-1 .. t-4
            const uint32_t row_base = (uint32_t)(16 * mt) << 16;
            for (int dl = 1; dl <= 4; ++dl) {
                const int l = t - dl;
                if (l < 0) break;
                const uint32_t col = (l >= st * TPS) ? 64 + 16 * (l % TPS) : 16 * (l % TPS);
                uint32_t r[8];
                ptx::tc_ld16_x2(tm + TM_G + col + row_base, r);
                ptx::tc_wait_ld();
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]) + 1.f;
                if (dl <= 2) {
                    uint4 a;
                    a.x = ptx::pack_bf16(-v[0], -v[1]);
                    a.y = ptx::pack_bf16(-v[2], -v[3]);
                    a.z = ptx::pack_bf16(-v[4], -v[5]);
                    a.w = ptx::pack_bf16(-v[6], -v[7]);
                    *reinterpret_cast<uint4 *>(s.cfrag[ps][mt][dl == 1 ? 1 : 0][lane]) = a;
                } else {
                    uint32_t a[4] = {ptx::pack_bf16(v[0], v[1]), ptx::pack_bf16(v[2], v[3]),
                                     ptx::pack_bf16(v[4], v[5]), ptx::pack_bf16(v[6], v[7])};
                    const int sel = lane >> 3, rr = lane & 7;
                    const uint32_t base = ptx::smem_addr(s.cb[ps][mt][dl == 4 ? 0 : 1]);
                    ptx::stsm_x4(base + ptx::sw32(rr + 8 * (sel & 1), sel >> 1), a);
                }
            }
        } else if (q == 2 + (mt >> 1)) {
            // Q_t rows: tril(Q_t K_t^T + 1) into rows 16 mt of the stage's output tile
            const uint32_t row_base = (uint32_t)(64 + 16 * mt) << 16;
            uint32_t r[8];
            ptx::tc_ld16_x2(tm + TM_G + 64 + 16 * mt + row_base, r);
            ptx::tc_wait_ld();
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int tt = g + 8 * ((i >> 1) & 1), ss = 2 * c + (i & 1) + 8 * (i >> 2);
                v[i] = ss <= tt ? __uint_as_float(r[i]) + 1.f : 0.f;
            }
            uint32_t a[4] = {ptx::pack_bf16(v[0], v[1]), ptx::pack_bf16(v[2], v[3]),
                             ptx::pack_bf16(v[4], v[5]), ptx::pack_bf16(v[6], v[7])};
            const int sel = lane >> 3, rr = lane & 7;
            ptx::stsm_x4(ptx::smem_addr(s.bout[ps]) + ptx::sw32(16 * mt + rr + 8 * (sel & 1), sel >> 1), a);
        }
        if (mt == TPS - 1 || t == N - 1) {
            ptx::fence_proxy_async();
            __syncwarp();
            ptx::tc_fence_before();
            if (lane == 0) ptx::mbar_arrive(bar_addr(&s.prep_full[ps]));
        }
    };

    for (int t = 0; t < min(N, 2 * TPS); ++t) prep(t);

    for (int n = 0; n < N; ++n) {
        // ---- W~_{n+1} (accumulator (n+1) % 2): bf16 operand tile, or the final state
        const int b = (n + 1) & 1;
        if (wait(&s.wupd_full[b], (n >> 1) & 1, n)) ptx::tc_fence_after();
        uint32_t wr[32], cr[4];
        ptx::tc_ld16_x8(tm + TM_W + 80 * b + lane_base, wr);
        ptx::tc_ld16_x1(tm + TM_W + 80 * b + 64 + lane_base, cr);
        ptx::tc_wait_ld();
        float w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __uint_as_float(wr[i]);
        const float c_lo = __uint_as_float(cr[0]), c_hi = __uint_as_float(cr[2]);
        if (n + 1 < N) {
            if (n >= 1) wait(&s.wbuf_free[b], ((n - 1) >> 1) & 1, n);
            write_wtile(b, w);
            write_bias(b, c_lo, c_hi);
            ptx::fence_proxy_async();
            __syncwarp();
            ptx::tc_fence_before();
            if (lane == 0) ptx::mbar_arrive(bar_addr(&s.wbuf_full[b]));
        } else {
            float *Wf = p.Wf + (size_t)bh * D * D;
            const int j0 = 16 * q + g, j1 = j0 + 8;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = 8 * k + 2 * c;
                Wf[i * D + j0] = w[4 * k];
                Wf[(i + 1) * D + j0] = w[4 * k + 1];
                Wf[i * D + j1] = w[4 * k + 2];
                Wf[(i + 1) * D + j1] = w[4 * k + 3];
            }
            if (c == 0) {
                p.bf[(size_t)bh * D + j0] = c_lo;
                p.bf[(size_t)bh * D + j1] = c_hi;
            }
        }
        if (n + 2 * TPS < N) prep(n + 2 * TPS);
    }
}

// Chain warps 0-3: quarter q owns output features 16q .. 16q + 15.
template <bool LN>
__device__ __forceinline__ void chain(Smem &s, const Params &p, uint32_t tm, int q, const Waiter &wait)
{
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int tid = threadIdx.x;   // 0..127
    const int N = p.N, h = blockIdx.x % p.H;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    // this thread's features: n-tile nt, element e: 16q + 8 nt + 2c + e
    float ga[2][2], be[2][2], g2[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 16 * q + 8 * nt + 2 * c + e;
            ga[nt][e] = LN ? p.gamma[(size_t)h * D + j] : 1.f;
            be[nt][e] = LN ? p.beta[(size_t)h * D + j] : 0.f;
            g2[nt][e] = ga[nt][e] * ga[nt][e];
        }
    float C1 = 0.f;
    if (LN)
        for (int j = 0; j < D; ++j) {
            const float gj = p.gamma[(size_t)h * D + j];
            C1 = fmaf(gj, gj, C1);
        }
    uint32_t gB1[4] = {0, 0, 0, 0}, gB2[4] = {0, 0, 0, 0};   // (eta G) B fragments of steps m-1, m-2
    float *xt = s.xtr[q];

    for (int m = 0; m < N; ++m) {
        const int st = m / TPS, mt = m % TPS, slot = st % NSS, ps = st % PS;
        if (mt == 0) {
            if (wait(&s.full[slot], (st / NSS) & 1, m)) {
            }
            wait(&s.prep_full[ps], (st / PS) & 1, m);
        }
        // ---- X''_m (features x tokens in TMEM) -> token-major fragments
        if (wait(&s.x_full[m % XR], (m / XR) & 1, m)) ptx::tc_fence_after();
        uint32_t xr[8];
        ptx::tc_ld16_x2(tm + TM_X + 16 * (m % XR) + lane_base, xr);
        ptx::tc_wait_ld();
        __syncwarp();
        xt[(2 * c) * 20 + g] = __uint_as_float(xr[0]);
        xt[(2 * c + 1) * 20 + g] = __uint_as_float(xr[1]);
        xt[(2 * c) * 20 + g + 8] = __uint_as_float(xr[2]);
        xt[(2 * c + 1) * 20 + g + 8] = __uint_as_float(xr[3]);
        xt[(8 + 2 * c) * 20 + g] = __uint_as_float(xr[4]);
        xt[(9 + 2 * c) * 20 + g] = __uint_as_float(xr[5]);
        xt[(8 + 2 * c) * 20 + g + 8] = __uint_as_float(xr[6]);
        xt[(9 + 2 * c) * 20 + g + 8] = __uint_as_float(xr[7]);
        __syncwarp();
        float pz[2][4];
        {
            const float2 a = *reinterpret_cast<const float2 *>(&xt[g * 20 + 2 * c]);
            const float2 b = *reinterpret_cast<const float2 *>(&xt[(g + 8) * 20 + 2 * c]);
            const float2 e = *reinterpret_cast<const float2 *>(&xt[g * 20 + 8 + 2 * c]);
            const float2 f = *reinterpret_cast<const float2 *>(&xt[(g + 8) * 20 + 8 + 2 * c]);
            pz[0][0] = a.x; pz[0][1] = a.y; pz[0][2] = b.x; pz[0][3] = b.y;
            pz[1][0] = e.x; pz[1][1] = e.y; pz[1][2] = f.x; pz[1][3] = f.y;
        }
        // ---- V (and K) of this mini-batch in the same fragment layout
        const int mrow = lane & 7, mat = lane >> 3;
        const int vrow = 16 * mt + mrow + 8 * (mat & 1), vchunk = 2 * q + (mat >> 1);
        uint32_t vr[4];
        ptx::ldsm_x4(ptx::smem_addr(s.stage[slot][2]) + ptx::sw128(vrow, vchunk), vr);
        float bp[2][4];   // LN: b' = gamma (beta - v + k);  plain: v
        if (LN) {
            uint32_t kr[4];
            ptx::ldsm_x4(ptx::smem_addr(s.stage[slot][0]) + ptx::sw128(vrow, vchunk), kr);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t vv = vr[2 * nt + hh], kk = kr[2 * nt + hh];
                    bp[nt][2 * hh] = ga[nt][0] * (be[nt][0] - ptx::bf16_lo(vv) + ptx::bf16_lo(kk));
                    bp[nt][2 * hh + 1] = ga[nt][1] * (be[nt][1] - ptx::bf16_hi(vv) + ptx::bf16_hi(kk));
                }
        } else {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    bp[nt][2 * hh] = ptx::bf16_lo(vr[2 * nt + hh]);
                    bp[nt][2 * hh + 1] = ptx::bf16_hi(vr[2 * nt + hh]);
                }
        }
        // ---- the two newest corrections: P -= C_{m,m-2} (eta G_{m-2}) + C_{m,m-1} (eta G_{m-1})
        if (m >= 2) {
            const uint4 a = *reinterpret_cast<const uint4 *>(s.cfrag[ps][mt][0][lane]);
            const uint32_t af[4] = {a.x, a.y, a.z, a.w};
            ptx::mma_bf16(pz[0], af, gB2[0], gB2[1]);
            ptx::mma_bf16(pz[1], af, gB2[2], gB2[3]);
        }
        if (m >= 1) {
            const uint4 a = *reinterpret_cast<const uint4 *>(s.cfrag[ps][mt][1][lane]);
            const uint32_t af[4] = {a.x, a.y, a.z, a.w};
            ptx::mma_bf16(pz[0], af, gB1[0], gB1[1]);
            ptx::mma_bf16(pz[1], af, gB1[2], gB1[3]);
        }
        // ---- G_m
        float gm[2][4];
        if (LN) {
            // per-token sums over this warp's 16 features, in fp32: partials over the
            // thread's 4 features, then a butterfly over the 4 lanes of the quad
            float sv[2][6];   // [token g / g+8][S1 z, S2 z^2, S3 g^2 z, S4 g^2 z^2, S5 b'z, S6 b']
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float a1 = 0.f, a2 = 0.f, a3 = 0.f, a4 = 0.f, a5 = 0.f, a6 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float z = pz[nt][2 * hh + e], b = bp[nt][2 * hh + e];
                        const float w = g2[nt][e] * z;
                        a1 += z;
                        a2 = fmaf(z, z, a2);
                        a3 += w;
                        a4 = fmaf(w, z, a4);
                        a5 = fmaf(b, z, a5);
                        a6 += b;
                    }
                sv[hh][0] = a1; sv[hh][1] = a2; sv[hh][2] = a3; sv[hh][3] = a4; sv[hh][4] = a5; sv[hh][5] = a6;
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int i = 0; i < 6; ++i) {
                    sv[hh][i] += __shfl_xor_sync(0xffffffffu, sv[hh][i], 1);
                    sv[hh][i] += __shfl_xor_sync(0xffffffffu, sv[hh][i], 2);
                }
            const int buf = m % 3;
            ptx::st_shared_f32(ptx::smem_addr(&s.stats[(m + 1) % 3][0][0]) + 4 * tid, 0.f);
            if (c == 0) {
                const uint32_t sb = ptx::smem_addr(&s.stats[buf][0][0]);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int i = 0; i < 6; ++i) ptx::red_add_shared(sb + 4 * ((g + 8 * hh) * 8 + i), sv[hh][i]);
            }
            ptx::named_bar(1, 128);
            float mu[2], al[2], bt[2], rr[2], de[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float4 a = *reinterpret_cast<const float4 *>(&s.stats[buf][g + 8 * hh][0]);
                const float2 b = *reinterpret_cast<const float2 *>(&s.stats[buf][g + 8 * hh][4]);
                const float S1 = a.x, S2 = a.y, S3 = a.z, S4 = a.w, S5 = b.x, S6 = b.y;
                const float inv_d = 1.f / D;
                const float u = S1 * inv_d;
                const float var = fmaxf(fmaf(S2, inv_d, -u * u), 0.f);
                const float r = rsqrtf(var + p.eps);
                const float A3 = fmaf(-u, C1, S3);
                const float A4 = fmaf(u * u, C1, fmaf(-2.f * u, S3, S4));
                const float A5 = fmaf(-u, S6, S5);
                const float m1 = fmaf(r, A3, S6) * inv_d;
                const float m2 = fmaf(r * r, A4, r * A5) * inv_d;
                mu[hh] = u;
                al[hh] = r * r;
                bt[hh] = r * r * m2;
                rr[hh] = r;
                de[hh] = r * m1;
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int hh = i >> 1, e = i & 1;
                    const float coef = fmaf(al[hh], g2[nt][e], -bt[hh]);
                    gm[nt][i] = fmaf(pz[nt][i] - mu[hh], coef, fmaf(rr[hh], bp[nt][i], -de[hh]));
                }
        } else {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) gm[nt][i] = pz[nt][i] - bp[nt][i];
        }
        // ---- eta G: B fragments for the next two steps, (eta G)^T tile for the tensor cores
        const float eg = s.eta[slot][16 * mt + g], eh = s.eta[slot][16 * mt + g + 8];
        uint32_t e4[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            e4[2 * nt] = ptx::pack_bf16(eg * gm[nt][0], eg * gm[nt][1]);
            e4[2 * nt + 1] = ptx::pack_bf16(eh * gm[nt][2], eh * gm[nt][3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            gB2[i] = gB1[i];
            gB1[i] = ptx::movm_t(e4[i]);
        }
        if (m >= GR) wait(&s.g_free[m % GR], ((m - GR) / GR) & 1, m);
        {
            const int sel = lane >> 3, rr = lane & 7;
            ptx::stsm_x4_t(ptx::smem_addr(s.gt[m % GR]) + ptx::sw32(16 * q + 8 * (sel >> 1) + rr, sel & 1), e4);
        }
        ptx::fence_proxy_async();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_addr(&s.g_full[m % GR]));
        if (mt == TPS - 1 || m == N - 1) {
            if (lane == 0) {
                ptx::mbar_arrive(bar_addr(&s.empty[slot]));
                ptx::mbar_arrive(bar_addr(&s.prep_free[ps]));
            }
        }
    }
}

// Epilogue warps 8-11: warp p finishes mini-batches n = p, p + 4, ...
template <bool LN>
__device__ __forceinline__ void epilogue(Smem &s, const Params &p, uint32_t tm, int pq,
                                         const CUtensorMap *tmZ, int bh, const Waiter &wait)
{
    const int lane = threadIdx.x & 31, c = lane & 3;
    const int N = p.N, h = bh % p.H;
    const uint32_t lane_base = (uint32_t)(32 * pq) << 16;
    float ga[16], be[16];
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 8 * k + 2 * c + e;
            ga[2 * k + e] = LN ? p.gamma[(size_t)h * D + j] : 1.f;
            be[2 * k + e] = LN ? p.beta[(size_t)h * D + j] : 0.f;
        }
    const uint32_t zb = ptx::smem_addr(s.zst[pq]);
    const int sel = lane >> 3, r8 = lane & 7;
    for (int n = pq; n < N; n += TPS) {
        const int st = n / TPS, slot = st % NSS;
        if (wait(&s.z_full[pq], (n / TPS) & 1, n)) ptx::tc_fence_after();
        uint32_t zr[32];
        ptx::tc_ld16_x8(tm + TM_Y + 64 * (n % YR) + lane_base, zr);
        ptx::tc_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_addr(&s.y_free[n % YR]));
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = __uint_as_float(zr[i]);
        float o[32];
        if (LN) {
            wait(&s.full[slot], (st / NSS) & 1, n);
            uint32_t qr[16];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                ptx::ldsm_x4(ptx::smem_addr(s.stage[slot][1]) +
                                 ptx::sw128(16 * pq + r8 + 8 * (sel & 1), 2 * i + (sel >> 1)),
                             qr + 4 * i);
            float s1[2] = {0.f, 0.f}, s2[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float a = z[4 * k + 2 * hh], b = z[4 * k + 2 * hh + 1];
                    s1[hh] += a + b;
                    s2[hh] = fmaf(a, a, fmaf(b, b, s2[hh]));
                }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                s1[hh] += __shfl_xor_sync(0xffffffffu, s1[hh], 1);
                s2[hh] += __shfl_xor_sync(0xffffffffu, s2[hh], 1);
                s1[hh] += __shfl_xor_sync(0xffffffffu, s1[hh], 2);
                s2[hh] += __shfl_xor_sync(0xffffffffu, s2[hh], 2);
            }
            float mu[2], r[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                mu[hh] = s1[hh] * (1.f / D);
                r[hh] = rsqrtf(fmaxf(fmaf(s2[hh], 1.f / D, -mu[hh] * mu[hh]), 0.f) + p.eps);
            }
            // q fragments: qr[4i + sel'] with sel' = (row half) + 2 (chunk parity); chunk k = 2i + (sel' >> 1)
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t qq = qr[4 * (k >> 1) + 2 * (k & 1) + hh];
                    const float q0 = ptx::bf16_lo(qq), q1 = ptx::bf16_hi(qq);
                    o[4 * k + 2 * hh] = q0 + fmaf(ga[2 * k] * (z[4 * k + 2 * hh] - mu[hh]), r[hh], be[2 * k]);
                    o[4 * k + 2 * hh + 1] =
                        q1 + fmaf(ga[2 * k + 1] * (z[4 * k + 2 * hh + 1] - mu[hh]), r[hh], be[2 * k + 1]);
                }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = z[i];
        }
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            pk[2 * k] = ptx::pack_bf16(o[4 * k], o[4 * k + 1]);
            pk[2 * k + 1] = ptx::pack_bf16(o[4 * k + 2], o[4 * k + 3]);
        }
        if (lane == 0) ptx::bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i)
            ptx::stsm_x4(zb + ptx::sw128(r8 + 8 * (sel & 1), 2 * i + (sel >> 1)), pk + 4 * i);
        ptx::fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
            ptx::tma_store_3d(tmZ, zb, 0, n * MB, bh);
            ptx::bulk_commit();
            ptx::mbar_arrive(bar_addr(&s.empty[slot]));
        }
    }
    if (lane == 0) ptx::bulk_wait<0>();
}

template <bool LN>
__global__ void __launch_bounds__(kThreads, 1)
linear_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmZ,
                    Params p)
{
    extern __shared__ unsigned char smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;

    if (tid == 0) {
        for (int i = 0; i < NSS; ++i) {
            ptx::mbar_init(bar_addr(&s.full[i]), 1);
            ptx::mbar_init(bar_addr(&s.empty[i]), 9);   // issuer + 4 chain + 4 epilogue
        }
        ptx::mbar_init(bar_addr(&s.gram_full), 1);
        for (int i = 0; i < PS; ++i) {
            ptx::mbar_init(bar_addr(&s.prep_full[i]), 4);
            ptx::mbar_init(bar_addr(&s.prep_free[i]), 5);   // 4 chain + issuer
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar_addr(&s.wbuf_full[i]), 4);
            ptx::mbar_init(bar_addr(&s.wbuf_free[i]), 1);
            ptx::mbar_init(bar_addr(&s.wupd_full[i]), 1);
        }
        for (int i = 0; i < XR; ++i) ptx::mbar_init(bar_addr(&s.x_full[i]), 1);
        for (int i = 0; i < GR; ++i) {
            ptx::mbar_init(bar_addr(&s.g_full[i]), 4);
            ptx::mbar_init(bar_addr(&s.g_free[i]), 1);
        }
        for (int i = 0; i < TPS; ++i) ptx::mbar_init(bar_addr(&s.z_full[i]), 1);
        for (int i = 0; i < YR; ++i) ptx::mbar_init(bar_addr(&s.y_free[i]), 1);
        ptx::mbar_init(bar_addr(&s.fin), 1);
        s.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp >= kAux0 && warp < kAux0 + 4) {
        // constant operand tiles: zeroed bias tiles, columns of ones
        const int t = tid - 32 * kAux0;   // 0..127
        uint32_t *ct = reinterpret_cast<uint32_t *>(s.ct);
        for (int i = t; i < 2 * D * MB / 2; i += 128) ct[i] = 0u;
        uint32_t *oa = reinterpret_cast<uint32_t *>(s.onesA);
        for (int i = t; i < ST * MB / 2; i += 128) oa[i] = 0u;
        uint32_t *ob = reinterpret_cast<uint32_t *>(s.onesB);
        for (int i = t; i < MB * MB / 2; i += 128) ob[i] = 0u;
        uint32_t *orr = reinterpret_cast<uint32_t *>(s.onesR);
        for (int i = t; i < MB * MB / 2; i += 128) orr[i] = 0u;
        float *st = &s.stats[0][0][0];
        for (int i = t; i < 3 * MB * 8; i += 128) st[i] = 0.f;
    }
    if (warp == kIssue) {
        ptx::tmem_alloc(ptx::smem_addr(&s.tmem), TM_COLS);
        ptx::tmem_relinquish();
    }
    __syncthreads();
    if (warp >= kAux0 && warp < kAux0 + 4) {
        const int t = tid - 32 * kAux0;
        const __nv_bfloat16 one = __float2bfloat16_rn(1.f);
        unsigned char *oa = reinterpret_cast<unsigned char *>(s.onesA);
        if (t < ST) *reinterpret_cast<__nv_bfloat16 *>(oa + ptx::sw32(t, 0)) = one;
        unsigned char *ob = reinterpret_cast<unsigned char *>(s.onesB);
        if (t < MB) *reinterpret_cast<__nv_bfloat16 *>(ob + ptx::sw32(t, 0)) = one;
        unsigned char *orr = reinterpret_cast<unsigned char *>(s.onesR);
        if (t < MB) *reinterpret_cast<__nv_bfloat16 *>(orr + ptx::sw32(0, t >> 3) + 2 * (t & 7)) = one;
        ptx::fence_proxy_async();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tm = s.tmem;
    const unsigned int role = warp < 4 ? 1u : warp < kEpi0 ? 2u : warp < kProd ? 3u : warp == kProd ? 4u : 5u;
    const Waiter wait{&s.abort_flag, p.status, p.wait_ns, s.full, role};

    if (warp < 4) {
        chain<LN>(s, p, tm, warp, wait);
    } else if (warp < kEpi0) {
        aux<LN>(s, p, tm, warp - kAux0, bh, wait);
    } else if (warp < kProd) {
        epilogue<LN>(s, p, tm, warp - kEpi0, &tmZ, bh, wait);
    } else if (warp == kProd) {
        if (lane == 0) producer(s, p, &tmK, &tmQ, &tmV, bh, wait);
    } else {
        if (lane == 0) issuer(s, p, tm, wait);
        __syncwarp();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kIssue) ptx::tmem_dealloc(tm, TM_COLS);
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
    Params p;
    p.H = d.H;
    p.L = d.L;
    p.N = d.L / MB;
    p.NST = (d.L + ST - 1) / ST;
    p.init_per_batch = d.init_per_batch;
    p.eps = d.ln_eps;
    p.wait_ns = g_wait_ns;
    p.withhold_loads = g_withhold_loads;
    p.eta = a.eta;
    p.W0 = a.W0;
    p.b0 = a.b0;
    p.gamma = a.gamma;
    p.beta = a.beta;
    p.Wf = a.W_final;
    p.bf = a.b_final;
    p.status = a.status;
    const size_t smem = sizeof(Smem) + 1024;
    auto kern = d.residual_ln ? linear_fused_kernel<true> : linear_fused_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<BH, kThreads, smem, a.stream>>>(mq, mk, mv, mz, p);
    return cudaGetLastError();
}

}  // namespace ttt
