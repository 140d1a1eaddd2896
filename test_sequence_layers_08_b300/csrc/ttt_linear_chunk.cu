// ttt_linear_chunk.cu -- TTT-Linear forward without the residual LayerNorm, bf16 I/O,
// d = 64, mini-batch b = 16: the fast weights are carried across chunks of 64 tokens
// (four mini-batches) instead of across single mini-batches.
//
// The method (damodev.csdn.net TTT article, sections 3.1 and 4.1-4.2): per (batch, head)
// the state S = [W; c] is updated once per mini-batch, every token's gradient taken at the
// mini-batch's starting state, and each output read with the state after its own token's
// update.  With the augmented rows k~ = [k, 1], q~ = [q, 1] and the squared-error loss
// (the no-LayerNorm inner model f(k) = k W + c):
//   G_m = K~_m S_m - V_m,   S_{m+1} = S_m - K~_m^T diag(eta_m) G_m.
// Unrolling four mini-batches m = 0..3 of a chunk from its starting state S gives, exactly,
//   G_m = (K~_m S - V_m) - sum_{l < m} L_{ml} G_l,   L_{ml}[t, s] = eta_s (k~_{m,t} . k~_{l,s})
//   Z    = Q~ S - (tril(Q~ K~^T) diag(eta)) G        (token-level causal, s <= t)
//   S'   = S - K~^T diag(eta) G                      (the whole chunk at once)
// i.e. the dual form of section 4.2 applied to a chunk of mini-batches, with the
// block-triangular correction L that keeps every gradient at its own mini-batch's state.
// With the inner-product loss -<f(k), v> of the ai-feeds Modular TTT page, G_m = -V_m.
// With its weight decay lambda (W only, the gradient at the mini-batch's start: inside
// mini-batch l, W_t = (1 - lambda cum_t) W_l - sum_{s<=t} eta_s k_s^T g_s, and
// W_{l+1} = d_l W_l - K_l^T E_l G_l with d_l = 1 - lambda sum_{s in l} eta_s), the unrolling stays
// exact with D_m = prod_{j<m} d_j and rho_{ml} = prod_{l<j<m} d_j:
//   G_m  = (D_m K_m W + 1 c - V_m) - sum_{l<m} [eta_s (rho_{ml} k_{m,t} . k_{l,s} + 1)] G_l
//   Z_t  = f_t D_m q_t W + c - sum_{l<m} [eta_s (f_t rho_{ml} q_t . k_{l,s} + 1)] G_l
//          - sum_{s in m, s<=t} eta_s (q_t . k_s + 1) g_s,          f_t = 1 - lambda cum_t
//   W'   = D_4 W - sum_l rho_{4l} K_l^T E_l G_l,  c' = c - sum_l G_l^T eta_l  (bias not decayed)
// (a template switch: the default learner pays none of it).
//
// B300 design.  The scan is latency-bound (one chunk of one (batch, head) waits on the
// last), so the kernel shortens the chain per token: the d x d state update, the key
// product of the next chunk and the query product of this one are 64-token warp-MMA
// GEMMs, and only the intra-chunk correction (three dependent 16 x 16 x 16 products)
// sits between them.  One CTA per (batch, head), eight warps in two roles:
//   * 64-token stages of Q, K, V (TMA, 128-byte swizzle) and eta (bulk copy) stream into
//     a 4-deep shared-memory ring; one thread refills a slot after the barrier that
//     retires it;
//   * state warps 0-3: warp w owns output features 16w..16w+15, its W^T rows live in
//     registers as fp32 accumulators; per chunk it forms G (P, Zbar, G are 16 x 64 register
//     tiles, features x tokens), runs the intra-chunk chain and the state update, then the
//     next chunk's key product and its six chain blocks L_{ml}; it publishes the chunk's
//     starting W^T (bf16 fragments) and -G through shared memory;
//   * output warps 4-7: one chunk behind, warp 4 + w forms Zbar for features 16w..16w+15:
//     the query product with the published starting state, the output corrections with the
//     published G, the Z tile (transposed with stmatrix into a swizzled staging tile and
//     written by a TMA store); it also computes the next chunk's ten output blocks.
//   So the state warps, whose chunk-to-chunk dependence is the critical path, issue only
//   the key side (about half of the per-chunk products), and the query side overlaps it;
//   the 16 x 16 blocks depend on the inputs alone and are shared as ready-made bf16 B
//   fragments through shared memory; one named barrier of all eight warps per chunk.
// Every mbarrier wait is bounded; a wait that runs out sets the library's failure flag
// and the kernel finishes without waiting again.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int D = 64;           // head dim
constexpr int MB = 16;          // mini-batch
constexpr int CT = 64;          // tokens per chunk (= per pipeline stage)
constexpr int NMB = CT / MB;    // mini-batches per chunk
constexpr int NSS = 4;          // stages in the ring (chunks i - 1, i, i + 1 are read in iteration i)
constexpr int kStateWarps = 4, kThreads = 256;
constexpr int kRefill = 96;     // thread that refills ring slots (a state warp)
constexpr int kStorer = 128;    // thread that stores Z tiles (an output warp)
constexpr uint32_t kTileBytes = CT * D * 2;   // 8 KB
constexpr int kBlocks = 16;     // 6 chain blocks + 10 output blocks

struct __align__(1024) Smem {
    __nv_bfloat16 q[NSS][CT * D];
    __nv_bfloat16 k[NSS][CT * D];
    __nv_bfloat16 v[NSS][CT * D];
    __nv_bfloat16 z[2][CT * D];
    uint2 blk[2][kBlocks][2][32];   // [chunk parity][block][source half][lane]
    uint4 ng[2][kStateWarps][NMB][32];   // -G_m A fragments [chunk parity][feature warp][m][lane]
    uint4 wa[2][kStateWarps][4][32];     // starting W^T A fragments [chunk parity][feature warp][k-step][lane]
    float2 cb[2][kStateWarps][32];       // starting c of the lane's features j0, j1
    float eta[NSS][CT];
    unsigned long long full[NSS];
    int abort_flag;
};

// Block numbering.  Chain block L_{ml} (m > l): (1,0) (2,0) (2,1) (3,0) (3,1) (3,2) -> 0..5.
// Output block (m, l), l <= m: 6 + m (m + 1) / 2 + l -> 6..15.
__host__ __device__ constexpr int chain_blk(int m, int l) { return m * (m - 1) / 2 + l; }
__host__ __device__ constexpr int out_blk(int m, int l) { return 6 + m * (m + 1) / 2 + l; }

struct Params {
    int H, L;
    long long wait_ns;       // bound of every mbarrier wait
    int withhold_loads;      // test hook: the producer issues no copies
    const float *eta, *W0, *b0;
    float *Wf, *bf;
    unsigned int *status;
    int init_per_batch;
    int hoff;                // head index of row 0 of this call
    int ip;                  // inner-product loss
    float wd;                // weight decay lambda (the WD instantiation)
};

constexpr long long kDrainNs = 1000000000ll;

__device__ __noinline__ bool chunk_wait_slow(uint32_t bar, uint32_t parity, long long limit,
                                             int *abort_flag, unsigned int *status)
{
    if (*(volatile int *)abort_flag) return false;
    if (ptx::mbar_wait_bounded(bar, parity, limit)) return true;
    *(volatile int *)abort_flag = 1;
    atomicOr(status, kStatusTimeout);
    return false;
}

template <bool WD>
__global__ void __launch_bounds__(kThreads, 1)
linear_chunk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmZ,
                    Params p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    Smem &s = *reinterpret_cast<Smem *>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, h = (p.hoff + bh) % p.H;
    const int NC = (p.L + CT - 1) / CT;   // chunks (= stages)

    const float *eta_bh = p.eta + (size_t)bh * p.L;
    auto issue_stage = [&](int st) {
        const int b = st % NSS, ntok = min(CT, p.L - st * CT);
        const uint32_t fb = ptx::smem_addr(&s.full[b]);
        ptx::mbar_arrive_expect_tx(fb, 3 * kTileBytes + ntok * 4);
        ptx::tma_load_3d(ptx::smem_addr(s.q[b]), &tmQ, fb, 0, st * CT, bh);
        ptx::tma_load_3d(ptx::smem_addr(s.k[b]), &tmK, fb, 0, st * CT, bh);
        ptx::tma_load_3d(ptx::smem_addr(s.v[b]), &tmV, fb, 0, st * CT, bh);
        ptx::bulk_load(ptx::smem_addr(s.eta[b]), eta_bh + st * CT, ntok * 4, fb);
    };
    const int nissue = p.withhold_loads ? 0 : NC;
    int issued = min(NSS, nissue);
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

    const int g = lane >> 2, c = lane & 3, mrow = lane & 7, mat = lane >> 3;
    const int fw = warp & 3;                         // feature group of this warp (both roles)
    const bool state_warp = warp < kStateWarps;
    const int j0 = fw * 16 + g, j1 = j0 + 8;         // this thread's two features
    bool aborted = false;

    auto wait_stage = [&](int st) {
        if (aborted) return;
        const uint32_t bar = ptx::smem_addr(&s.full[st % NSS]);
        if (ptx::mbar_try_wait(bar, (st / NSS) & 1)) return;
        aborted = !chunk_wait_slow(bar, (st / NSS) & 1, p.wait_ns, &s.abort_flag, p.status);
    };
    // byte address of token row t, 16-byte chunk ch of the stage tile of chunk cc; callers
    // pass t = 8 k + mrow, so the swizzle term is (ch ^ mrow)
    auto tile_addr = [&](const __nv_bfloat16 (*arr)[CT * D], int cc, int t, int ch) -> uint32_t {
        return ptx::smem_addr(arr[cc % NSS]) + (uint32_t)(t * 128 + ((ch ^ mrow) << 4));
    };
    // eta of tokens t, t + 1 (t even) of chunk cc
    auto eta2 = [&](int cc, int t) -> float2 {
        return *reinterpret_cast<const float2 *>(&s.eta[cc % NSS][t]);
    };
    // the slot of a ragged last stage holds stale eta past the sequence: every warp zeroes it
    // (identical values) before its own first read of that stage
    const int tail = p.L - (NC - 1) * CT;
    auto zero_eta_tail = [&](int cc) {
        if (cc == NC - 1 && tail < CT) {
            for (int t = tail + lane; t < CT; t += 32) s.eta[cc % NSS][t] = 0.f;
            __syncwarp();
        }
    };

    // ---- initial state (state warps): W^T rows j0/j1 as fp32 accumulators, c
    float wt[8][4];
    float cb0 = 0.f, cb1 = 0.f;
    const size_t init = p.init_per_batch ? (size_t)bh : (size_t)h;
    if (state_warp) {
        const float *W0 = p.W0 + init * D * D;
#pragma unroll
        for (int pt = 0; pt < 8; ++pt) {
            const int i = pt * 8 + 2 * c;
            wt[pt][0] = W0[i * D + j0];
            wt[pt][1] = W0[(i + 1) * D + j0];
            wt[pt][2] = W0[i * D + j1];
            wt[pt][3] = W0[(i + 1) * D + j1];
        }
        cb0 = p.b0[init * D + j0];
        cb1 = p.b0[init * D + j1];
    }
    const float kf = p.ip ? 0.f : 1.f;   // weight of P in G (0: inner-product loss, G = -V)

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

    // acc[nt] = W^T X^T + c over the 64 tokens of chunk cc (n-tile nt = tokens 8 nt..8 nt + 7)
    auto product = [&](float (*acc)[4], const __nv_bfloat16 (*arr)[CT * D], int cc, float c0, float c1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int tb = 0; tb < 4; ++tb) {
                // matrices: (t-block 2 tb, chunk 2q), (2 tb, 2q + 1), (2 tb + 1, 2q), (2 tb + 1, 2q + 1)
                uint32_t r[4];
                ptx::ldsm_x4(tile_addr(arr, cc, (2 * tb + (mat >> 1)) * 8 + mrow, 2 * q + (mat & 1)), r);
                if (q == 0) {
                    ptx::mma_bf16_c(acc[2 * tb], wa[q], r[0], r[1], c0, c0, c1, c1);
                    ptx::mma_bf16_c(acc[2 * tb + 1], wa[q], r[2], r[3], c0, c0, c1, c1);
                } else {
                    ptx::mma_bf16(acc[2 * tb], wa[q], r[0], r[1]);
                    ptx::mma_bf16(acc[2 * tb + 1], wa[q], r[2], r[3]);
                }
            }
        }
    };

    // Input-only block: rows t = target tokens of mini-batch mt of X (Q or K), columns s =
    // source tokens of mini-batch l of K; value eta_s (x_t . k_s + 1), masked to s <= t on a
    // diagonal output block.  Stored as the lane's own B fragments (k = s, n = t).
    // With weight decay the Gram part of rows t = g (t = g + 8) is scaled by sc0 (sc1).
    auto block = [&](const __nv_bfloat16 (*X)[CT * D], int cc, int mt, int l, bool causal, int b, float sc0,
                     float sc1) {
        uint32_t a[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q)   // A: matrices (t0, ch 2q), (t1, 2q), (t0, 2q + 1), (t1, 2q + 1)
            ptx::ldsm_x4(tile_addr(X, cc, mt * MB + (mat & 1) * 8 + mrow, 2 * q + (mat >> 1)), a[q]);
        float acc[2][4], ac2[2][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // B: source rows s: matrices (half 0, ch 2q), (half 0, 2q + 1), (half 1, 2q), (half 1, 2q + 1)
            uint32_t r[4];
            ptx::ldsm_x4(tile_addr(s.k, cc, l * MB + (mat >> 1) * 8 + mrow, 2 * q + (mat & 1)), r);
            float (*dst)[4] = (q & 1) ? ac2 : acc;
            if (q < 2) {
                ptx::mma_bf16_c(dst[0], a[q], r[0], r[1], 0.f, 0.f, 0.f, 0.f);
                ptx::mma_bf16_c(dst[1], a[q], r[2], r[3], 0.f, 0.f, 0.f, 0.f);
            } else {
                ptx::mma_bf16(dst[0], a[q], r[0], r[1]);
                ptx::mma_bf16(dst[1], a[q], r[2], r[3]);
            }
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            // rows t = g, g + 8; columns s = 8 hf + 2c, +1
            const int s0 = hf * 8 + 2 * c;
            const float2 e = eta2(cc, l * MB + s0);
            const float e0 = e.x, e1 = e.y;
            float x0 = acc[hf][0] + ac2[hf][0], x1 = acc[hf][1] + ac2[hf][1];
            float x2 = acc[hf][2] + ac2[hf][2], x3 = acc[hf][3] + ac2[hf][3];
            if (WD) {
                x0 *= sc0;
                x1 *= sc0;
                x2 *= sc1;
                x3 *= sc1;
            }
            const float v0 = (causal && s0 > g) ? 0.f : e0 * (x0 + 1.f);
            const float v1 = (causal && s0 + 1 > g) ? 0.f : e1 * (x1 + 1.f);
            const float v2 = (causal && s0 > g + 8) ? 0.f : e0 * (x2 + 1.f);
            const float v3 = (causal && s0 + 1 > g + 8) ? 0.f : e1 * (x3 + 1.f);
            s.blk[cc & 1][b][hf][lane] = make_uint2(ptx::pack_bf16(v0, v1), ptx::pack_bf16(v2, v3));
        }
    };
    // Weight decay.  An inclusive scan of eta within each mini-batch of chunk cc: lane l holds the
    // prefix sums at tokens l and l + 32 (mini-batches l / 16 and 2 + l / 16).  The mini-batch
    // factors d_l = 1 - lambda sum eta are the segment ends; rho_{ml} = prod_{l<j<m} d_j; the
    // query factor of token t of mini-batch m is one shuffle away.
    struct EtaScan {
        float ca, cb;
    };
    auto eta_scan = [&](int cc, float *dl) -> EtaScan {
        zero_eta_tail(cc);
        float a = s.eta[cc % NSS][lane], b2 = s.eta[cc % NSS][lane + 32];
#pragma unroll
        for (int o = 1; o < MB; o <<= 1) {
            const float ta = __shfl_up_sync(0xffffffffu, a, o, MB), tb = __shfl_up_sync(0xffffffffu, b2, o, MB);
            if ((lane & (MB - 1)) >= o) {
                a += ta;
                b2 += tb;
            }
        }
        dl[0] = 1.f - p.wd * __shfl_sync(0xffffffffu, a, MB - 1);
        dl[1] = 1.f - p.wd * __shfl_sync(0xffffffffu, a, 2 * MB - 1);
        dl[2] = 1.f - p.wd * __shfl_sync(0xffffffffu, b2, MB - 1);
        dl[3] = 1.f - p.wd * __shfl_sync(0xffffffffu, b2, 2 * MB - 1);
        return EtaScan{a, b2};
    };
    auto rho = [&](const float *dl, int m, int l) {
        float r = 1.f;
#pragma unroll
        for (int j = 0; j < NMB; ++j)
            if (j > l && j < m) r *= dl[j];
        return r;
    };
    // 1 - lambda cum_t for token t of mini-batch m (m uniform across the warp; every lane shuffles)
    auto fq_tok = [&](const EtaScan &es, int m, int t) {
        const int idx = (m * MB + t) & 31;
        const float va = __shfl_sync(0xffffffffu, es.ca, idx), vb = __shfl_sync(0xffffffffu, es.cb, idx);
        return 1.f - p.wd * (m < 2 ? va : vb);
    };
    // P (or the query product) of mini-batch m from the product without bias: f D_m x + c
    auto scale_rows = [&](float (*acc)[4], const float *dl, const EtaScan &es, bool per_token, float c0, float c1) {
        float Dm = 1.f;
#pragma unroll
        for (int m = 0; m < NMB; ++m) {
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float f = (per_token ? fq_tok(es, m, 8 * u + 2 * c + e) : 1.f) * Dm;
                    acc[2 * m + u][e] = fmaf(f, acc[2 * m + u][e], c0);
                    acc[2 * m + u][2 + e] = fmaf(f, acc[2 * m + u][2 + e], c1);
                }
            Dm *= dl[m];
        }
    };
    // chain blocks L_{ml} (m > l; numbers 0..5) of chunk cc: state warp w takes those with
    // number = w mod 4
    auto chain_blocks = [&](int cc) {
        zero_eta_tail(cc);
        float dl[NMB] = {1.f, 1.f, 1.f, 1.f};
        if (WD) eta_scan(cc, dl);
#pragma unroll
        for (int m = 1; m < NMB; ++m)
#pragma unroll
            for (int l = 0; l < m; ++l)
                if (chain_blk(m, l) % kStateWarps == fw) {
                    const float r = WD ? rho(dl, m, l) : 1.f;
                    block(s.k, cc, m, l, false, chain_blk(m, l), r, r);
                }
    };
    // output blocks (m, l), l <= m (numbers 6..15) of chunk cc: output warp 4 + w takes those
    // with (number - 6) = w mod 4
    auto out_blocks = [&](int cc) {
        zero_eta_tail(cc);
        float dl[NMB] = {1.f, 1.f, 1.f, 1.f};
        EtaScan es{0.f, 0.f};
        if (WD) es = eta_scan(cc, dl);
#pragma unroll
        for (int m = 0; m < NMB; ++m)
#pragma unroll
            for (int l = 0; l <= m; ++l)
                if ((out_blk(m, l) - 6) % kStateWarps == fw) {
                    // earlier mini-batches: f_t rho_{ml} on the Gram part; the diagonal block: none
                    float s0 = 1.f, s1 = 1.f;
                    if (WD && l < m) {
                        const float r = rho(dl, m, l);
                        s0 = r * fq_tok(es, m, g);
                        s1 = r * fq_tok(es, m, g + 8);
                    }
                    block(s.q, cc, m, l, l == m, out_blk(m, l), s0, s1);
                }
    };
    // both n-tiles of a block: (f0.x, f1.x) for target tokens 0-7, (f0.y, f1.y) for 8-15
    auto read_blk = [&](int cc, int b, uint2 &f0, uint2 &f1) {
        f0 = s.blk[cc & 1][b][0][lane];
        f1 = s.blk[cc & 1][b][1][lane];
    };

    // ---- prologue (state warps): P_0 = K_0 W_0 + c_0 and the chain blocks of chunk 0
    float pacc[8][4];
    if (state_warp) {
        wait_stage(0);
        pack_w();
        if (WD) {
            float dl[NMB];
            const EtaScan es = eta_scan(0, dl);
            product(pacc, s.k, 0, 0.f, 0.f);
            scale_rows(pacc, dl, es, false, cb0, cb1);
        } else {
            product(pacc, s.k, 0, cb0, cb1);
        }
        chain_blocks(0);
    }
    ptx::named_bar(1, kThreads);   // every state warp reads all six chain blocks of chunk 0

    // Iteration i: the state warps run chunk i (i < NC); the output warps compute the output
    // blocks of chunk i (i < NC) and the outputs of chunk i - 1 (i >= 1).  The barrier at the
    // end of the iteration publishes both; stage i - 1 is then no longer read.
    for (int it = 0; it <= NC; ++it) {
        if (state_warp && it < NC) {
            const int cc = it;
            const bool more = cc + 1 < NC;
            if (more) wait_stage(cc + 1);
            // the chunk's starting state for the output warps
#pragma unroll
            for (int q = 0; q < 4; ++q) s.wa[cc & 1][fw][q][lane] = make_uint4(wa[q][0], wa[q][1], wa[q][2], wa[q][3]);
            s.cb[cc & 1][fw][lane] = make_float2(cb0, cb1);

            // weight decay: W' = D_4 W - sum_m rho_{4m} K_m^T E_m G_m (the carried W^T scaled first)
            float dl[NMB] = {1.f, 1.f, 1.f, 1.f};
            if (WD) {
                eta_scan(cc, dl);
                const float D4 = dl[0] * dl[1] * dl[2] * dl[3];
#pragma unroll
                for (int pt = 0; pt < 8; ++pt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) wt[pt][i] *= D4;
            }

            // intra-chunk chain: G_m, then its corrections to the later mini-batches' P and its
            // k-step of the state update
            float d0 = 0.f, d1 = 0.f;   // eta^T G for features j0, j1 (this thread's tokens)
#pragma unroll
            for (int m = 0; m < NMB; ++m) {
                float vt[2][4];
                {
                    uint32_t r[4];   // V^T of mini-batch m: matrices (t0, j0), (t0, j1), (t1, j0), (t1, j1)
                    ptx::ldsm_x4_t(tile_addr(s.v, cc, m * MB + (mat >> 1) * 8 + mrow, fw * 2 + (mat & 1)), r);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        vt[u][0] = ptx::bf16_lo(r[2 * u]);
                        vt[u][1] = ptx::bf16_hi(r[2 * u]);
                        vt[u][2] = ptx::bf16_lo(r[2 * u + 1]);
                        vt[u][3] = ptx::bf16_hi(r[2 * u + 1]);
                    }
                }
                float gm[2][4];
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) gm[u][i] = fmaf(pacc[2 * m + u][i], kf, -vt[u][i]);
                uint32_t ng[4];
                ng[0] = ptx::pack_bf16(-gm[0][0], -gm[0][1]);
                ng[1] = ptx::pack_bf16(-gm[0][2], -gm[0][3]);
                ng[2] = ptx::pack_bf16(-gm[1][0], -gm[1][1]);
                ng[3] = ptx::pack_bf16(-gm[1][2], -gm[1][3]);
                s.ng[cc & 1][fw][m][lane] = make_uint4(ng[0], ng[1], ng[2], ng[3]);
                // chain: P_{m'} -= G_m L_{m'm}^T for the later mini-batches
#pragma unroll
                for (int mp = m + 1; mp < NMB; ++mp) {
                    uint2 f0, f1;
                    read_blk(cc, chain_blk(mp, m), f0, f1);
                    ptx::mma_bf16(pacc[2 * mp], ng, f0.x, f1.x);
                    ptx::mma_bf16(pacc[2 * mp + 1], ng, f0.y, f1.y);
                }
                // state update, k-step m: W^T += (-eta G_m)^T K_m
                const int s0 = m * MB + 2 * c;
                const float2 ea = eta2(cc, s0), eb = eta2(cc, s0 + 8);
                const float e00 = ea.x, e01 = ea.y, e10 = eb.x, e11 = eb.y;
                uint32_t nge[4];
                const float r4 = WD ? rho(dl, NMB, m) : 1.f;   // rho_{4m}
                nge[0] = ptx::pack_bf16(-r4 * e00 * gm[0][0], -r4 * e01 * gm[0][1]);
                nge[1] = ptx::pack_bf16(-r4 * e00 * gm[0][2], -r4 * e01 * gm[0][3]);
                nge[2] = ptx::pack_bf16(-r4 * e10 * gm[1][0], -r4 * e11 * gm[1][1]);
                nge[3] = ptx::pack_bf16(-r4 * e10 * gm[1][2], -r4 * e11 * gm[1][3]);
                d0 += e00 * gm[0][0] + e01 * gm[0][1] + e10 * gm[1][0] + e11 * gm[1][1];
                d1 += e00 * gm[0][2] + e01 * gm[0][3] + e10 * gm[1][2] + e11 * gm[1][3];
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    // matrices (s-block, i-chunk): (0, 2pp), (1, 2pp), (0, 2pp + 1), (1, 2pp + 1)
                    uint32_t r[4];
                    ptx::ldsm_x4_t(tile_addr(s.k, cc, m * MB + (mat & 1) * 8 + mrow, 2 * pp + (mat >> 1)), r);
                    ptx::mma_bf16(wt[2 * pp], nge, r[0], r[1]);
                    ptx::mma_bf16(wt[2 * pp + 1], nge, r[2], r[3]);
                }
            }
            // c -= eta^T G over the chunk (sum over the four lanes sharing g)
            d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
            d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
            cb0 -= d0;
            cb1 -= d1;
            pack_w();

            // next chunk: its key product from the new state, and its chain blocks
            if (more) {
                if (WD) {
                    float dn[NMB];
                    const EtaScan es = eta_scan(cc + 1, dn);
                    product(pacc, s.k, cc + 1, 0.f, 0.f);
                    scale_rows(pacc, dn, es, false, cb0, cb1);
                } else {
                    product(pacc, s.k, cc + 1, cb0, cb1);
                }
                chain_blocks(cc + 1);
            }
        } else if (!state_warp) {
            if (it < NC) {
                wait_stage(it);
                out_blocks(it);
            }
            if (it >= 1) {
                const int cc = it - 1;
                // query-side product with the chunk's starting state (published by the state warp
                // of the same features)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w4 = s.wa[cc & 1][fw][q][lane];
                    wa[q][0] = w4.x;
                    wa[q][1] = w4.y;
                    wa[q][2] = w4.z;
                    wa[q][3] = w4.w;
                }
                const float2 cbs = s.cb[cc & 1][fw][lane];
                float yacc[8][4];
                if (WD) {   // token t of mini-batch m reads f_t D_m W (and c, not decayed)
                    float dl[NMB];
                    const EtaScan es = eta_scan(cc, dl);
                    product(yacc, s.q, cc, 0.f, 0.f);
                    scale_rows(yacc, dl, es, true, cbs.x, cbs.y);
                } else {
                    product(yacc, s.q, cc, cbs.x, cbs.y);
                }
                // outputs: Zbar_{m'} -= G_m B_{m'm}^T for m' >= m
#pragma unroll
                for (int m = 0; m < NMB; ++m) {
                    const uint4 n4 = s.ng[cc & 1][fw][m][lane];
                    const uint32_t ng[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
                    for (int mp = m; mp < NMB; ++mp) {
                        uint2 f0, f1;
                        read_blk(cc, out_blk(mp, m), f0, f1);
                        ptx::mma_bf16(yacc[2 * mp], ng, f0.x, f1.x);
                        ptx::mma_bf16(yacc[2 * mp + 1], ng, f0.y, f1.y);
                    }
                }
                // Zbar -> bf16 staging tile cc % 2 (rows = tokens), TMA-stored after the barrier
                const uint32_t zaddr = ptx::smem_addr(s.z[cc & 1]);
#pragma unroll
                for (int m = 0; m < NMB; ++m) {
                    uint32_t r[4];
                    r[0] = ptx::pack_bf16(yacc[2 * m][0], yacc[2 * m][1]);
                    r[1] = ptx::pack_bf16(yacc[2 * m][2], yacc[2 * m][3]);
                    r[2] = ptx::pack_bf16(yacc[2 * m + 1][0], yacc[2 * m + 1][1]);
                    r[3] = ptx::pack_bf16(yacc[2 * m + 1][2], yacc[2 * m + 1][3]);
                    // matrices (j-block, t-block): (0,0), (1,0), (0,1), (1,1)
                    ptx::stsm_x4_t(zaddr + ptx::sw128(m * MB + (mat >> 1) * 8 + mrow, fw * 2 + (mat & 1)), r);
                }
                ptx::fence_proxy_async();
            }
            // the store of chunk it - 2 has read its tile (which chunk it overwrites next)
            if (tid == kStorer) ptx::bulk_wait_read<0>();
        }
        ptx::named_bar(1, kThreads);
        if (tid == kStorer && it >= 1) {
            ptx::tma_store_3d(&tmZ, ptx::smem_addr(s.z[(it - 1) & 1]), 0, (it - 1) * CT, bh);
            ptx::bulk_commit();
        }
        if (tid == kRefill && it >= 1 && it - 1 + NSS < nissue && !aborted) {
            // stage it - 1 is no longer read: refill its slot with stage it - 1 + NSS
            ptx::fence_proxy_async();
            issue_stage(it - 1 + NSS);
            issued = it - 1 + NSS + 1;
        }
    }
    if (tid == kStorer) ptx::bulk_wait<0>();
    if (tid == kRefill)   // copies still in flight (only after a wait ran out) land before exit
        for (int st = max(0, issued - NSS); st < issued; ++st)
            ptx::mbar_wait_bounded(ptx::smem_addr(&s.full[st % NSS]), (st / NSS) & 1, kDrainNs);
    if (state_warp) {
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

}  // namespace

bool linear_chunk_supported(const ttt_desc &d)
{
    return d.io_dtype == TTT_BF16 && d.d == D && d.mini_batch == MB && !d.residual_ln;
}

cudaError_t launch_linear_chunk(const LinearArgs &a)
{
    const ttt_desc &d = a.desc;
    const int BH = call_rows(d);
    CUtensorMap mq, mk, mv, mz;
    if (!make_bf16_tile_map(&mq, a.Q, d.L, BH, CT) || !make_bf16_tile_map(&mk, a.K, d.L, BH, CT) ||
        !make_bf16_tile_map(&mv, a.V, d.L, BH, CT) || !make_bf16_tile_map(&mz, a.Z, d.L, BH, CT))
        return cudaErrorInvalidValue;
    Params p{d.H, d.L, wait_timeout_ns(), withhold_loads(), a.eta, a.W0, a.b0, a.W_final, a.b_final,
             a.status, d.init_per_batch, head_offset(d), d.loss == TTT_LOSS_INNER_PRODUCT, d.weight_decay};
    const size_t smem = sizeof(Smem) + 1024;
    const auto kern = d.weight_decay != 0.f ? linear_chunk_kernel<true> : linear_chunk_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<BH, kThreads, smem, a.stream>>>(mq, mk, mv, mz, p);
    return cudaGetLastError();
}

}  // namespace ttt
