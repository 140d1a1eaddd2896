// ttt_mlp_tmem.cu -- TTT-MLP forward with the hidden-width products on tcgen05 and the fast
// weights resident in tensor memory (bf16 I/O, d = 64, d_hidden = 256, b = 16, no weight decay).
//
// The method is the one of the warp-MMA kernel (TTT-MLP of the lryc.cn TTT article, section
// 2.1; mini-batch gradient descent of the damodev.csdn.net TTT article, sections 4.1-4.2).
// Per (batch, head) and mini-batch n of 16 tokens, with the weights of the mini-batch start
// on every right-hand side:
//   Z1 = K W1 + b1,  X2 = GELU(Z1),  Z2 = X2 W2 + b2
//   G2 = LNbwd(Z2; V - K)  (or kf Z2 - V without the LayerNorm),  G1 = (G2 W2^T) . GELU'(Z1)
//   W1 -= K^T diag(eta) G1,  b1 -= eta^T G1,  W2 -= X2^T diag(eta) G2,  b2 -= eta^T G2
//   Zb1 = Q W1 + b1 - (eta_s (q_t . k_s + 1) [s <= t]) G1,   Xb2 = GELU(Zb1)
//   Zb2 = Xb2 W2 + b2 - (eta_s (xb2_t . x2_s + 1) [s <= t]) G2,   Z = Q + LN(Zb2)
//
// B300 design.  The products run transposed, the 256 hidden units as the MMA's M (two
// 128-lane halves) and the tokens as N, so that W1^T and W2 live in tensor memory as fp32
// accumulators which the updates add into (no round trip of the state through registers):
//   TMEM columns  W1^T [h][i] 0-127 | W2 [h][o] 128-255 | Z1^T key, query 256-319 |
//                 G1^T 320-351 | Z2^T 352-367 (lanes = outputs) | Zb2^T 368-399 (by parity)
//   one thread of the control warp issues, per mini-batch, five groups (one commit each):
//     M1  Z1^T = W1^T [K | Q]^T     A: bf16 copy of W1^T          B: the K, Q rows as TMA writes them
//     M2  Z2^T = W2^T X2^T          A: bf16 W2^T, outputs padded to 128 rows by reading on
//                                      into the next block       B: X2 [t][h]
//     M3  G1^T = W2 G2^T            A: bf16 copy of W2            B: G2 [t][o]
//     M4  W1^T += (-eta G1)^T K,  W2 += X2^T (-eta G2),  Zb1^T += (-eta G1)^T A1^T
//     M5  Zb2^T = W2^T Xb2^T + (-eta G2)^T A2^T
//   eight compute warps, thread = hidden unit (warp group = half, warp = lane quadrant),
//   turn each result into the next operand: GELU and GELU' of Z1 (X2 as a [t][h] column and
//   an [h][t] row), G1 . GELU', Xb2, and after M4 the bf16 copies of the updated weights
//   (W1^T, W2 rows; W2^T a column at a time once M5 has read the old one).  Warps 0-3 run
//   both LayerNorms on the 64 outputs of the 16 tokens (Z2^T moved through shared memory,
//   eight threads per token); the output LayerNorm of mini-batch n runs while M2 of n + 1 is
//   in flight.  Warp 5 builds K^T and A1 = (q_t . k_s + 1) [s <= t] one mini-batch ahead;
//   warps 6-7 the Gram A2 = (xb2_t . x2_s + 1) [s <= t] (warp MMA over the hidden halves);
//   eta is folded into -eta G, so neither block carries it.
// Every operand is K-major with the 128-byte swizzle; operands 16 tokens deep use the first
// 32 bytes of each 128-byte row (one K16 step).  Every mbarrier wait is bounded: after one runs
// out, the control thread stops issuing and the compute warps run the rest of the scan
// without waiting (their named barriers stay matched), the outputs are garbage and the
// failure flag is set.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int D = 64;            // model / head dim
constexpr int DH = 256;          // hidden dim
constexpr int MB = 16;           // mini-batch
constexpr int ST = 64;           // tokens per pipeline stage
constexpr int TPS = ST / MB;     // mini-batches per stage
constexpr int NSS = 2;           // stages in the ring
constexpr int kCompute = 8;      // compute warps
constexpr int kCtl = 8;          // control warp (TMEM owner; lane 0 issues copies and MMAs)
constexpr int kThreads = (kCompute + 1) * 32;
constexpr int kPrepWarp = 5;     // K^T and A1, one mini-batch ahead
constexpr int kGramWarp = 6;     // A2 (with warp 7)
constexpr int kBarLn = 2, kBarGram = 3;
constexpr uint32_t kStageTileBytes = ST * D * 2;   // 8 KB
constexpr uint32_t cW1 = 0, cW2 = 128, cZ1 = 256, cG1 = 320, cZ2 = 352, cZB2 = 368, kTmemCols = 512;
constexpr uint32_t kI16 = ptx::idesc_bf16_kk(128, 16), kI64 = ptx::idesc_bf16_kk(128, 64);
constexpr long long kDrainNs = 1000000000ll;

struct __align__(1024) Smem {
    unsigned char q[NSS][kStageTileBytes];   // [token][i], 128-byte rows, TMA 128-byte swizzle
    unsigned char k[NSS][kStageTileBytes];
    unsigned char v[NSS][kStageTileBytes];
    unsigned char w1t[DH * 128];             // W1^T [h][i]
    unsigned char w2t[4][D * 128];           // W2^T [o][h], one 64-row block per 64 hidden units
    unsigned char w2[DH * 128];              // W2 [h][o]; follows w2t (M2 reads 128-row blocks)
    unsigned char upd[DH * 128];             // [h][s]: columns 0-15 -eta G1, 16-31 X2
    unsigned char kte[128 * 128];            // [i|o][s]: columns 0-15 K^T, 16-31 (-eta G2)^T; rows 64+ zero
    unsigned char x2[4][MB * 128];           // X2 [t][h], one block per 64 hidden units
    unsigned char xb2[4][MB * 128];          // Xb2 [t][h]
    unsigned char g2[MB * 128];              // G2 [t][o]
    unsigned char a1[MB * 128];              // A1 [t][s] (columns 0-15)
    unsigned char a2[MB * 128];              // A2 [t][s]
    unsigned char zst[MB * 128];             // output staging [t][o]
    float zb[MB][68];                        // Z2 then -eta G2, or Zb2 [t][o] (fp32)
    float gram[32][8];                       // warp 7's half of the Gram
    float eta[NSS][ST];
    unsigned long long full[NSS], empty[NSS], mma[5];
    unsigned long long x2r, g2r, g1r, xbr, prep, a2r, init, drain;
    uint32_t tmem;
    int abort_flag;
};
static_assert(offsetof(Smem, w2) == offsetof(Smem, w2t) + 4 * D * 128, "w2 directly follows w2t");
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");

struct Params {
    int H, L, N, NST, init_per_batch;
    float eps;
    long long wait_ns;
    int withhold_loads;
    const float *eta, *W1, *b1, *W2, *b2, *gamma, *beta;
    float *W1f, *b1f, *W2f, *b2f;
    unsigned int *status;
    int hoff;   // head index of row 0 of this call
    int ip;     // inner-product loss
};

__device__ __noinline__ bool tmem_wait_slow(uint32_t bar, uint32_t parity, long long limit, int *abort_flag,
                                            unsigned int *status)
{
    if (*(volatile int *)abort_flag) return false;
    if (ptx::mbar_wait_bounded(bar, parity, limit)) return true;
    *(volatile int *)abort_flag = 1;
    atomicOr(status, kStatusTimeout);
    return false;
}

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

__device__ __forceinline__ uint16_t bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ uint4 pack8(const float *v)
{
    return make_uint4(ptx::pack_bf16(v[0], v[1]), ptx::pack_bf16(v[2], v[3]), ptx::pack_bf16(v[4], v[5]),
                      ptx::pack_bf16(v[6], v[7]));
}
__device__ __forceinline__ void unpack8(uint4 u, float *v)
{
    v[0] = ptx::bf16_lo(u.x); v[1] = ptx::bf16_hi(u.x);
    v[2] = ptx::bf16_lo(u.y); v[3] = ptx::bf16_hi(u.y);
    v[4] = ptx::bf16_lo(u.z); v[5] = ptx::bf16_hi(u.z);
    v[6] = ptx::bf16_lo(u.w); v[7] = ptx::bf16_hi(u.w);
}
// element (row, col) of a 128-byte-swizzled bf16 tile (col < 64)
__device__ __forceinline__ uint32_t el(int row, int col) { return ptx::sw128(row, col >> 3) + ((col & 7) << 1); }
__device__ __forceinline__ uint64_t dsc(uint32_t addr) { return ptx::sdesc_sw128(addr); }

template <bool LN>
__global__ void __launch_bounds__(kThreads, 1)
mlp_tmem_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmZ, Params p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    Smem &s = *reinterpret_cast<Smem *>(smem_raw + (((raw + 1023u) & ~1023u) - raw));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, head = (p.hoff + bh) % p.H;
    const int N = p.N;
    auto A = [](const void *ptr) { return ptx::smem_addr(ptr); };

    const float *eta_bh = p.eta + (size_t)bh * p.L;
    auto issue_stage = [&](int st) {
        const int b = st % NSS, ntok = min(ST, p.L - st * ST);
        const uint32_t fb = A(&s.full[b]);
        ptx::mbar_arrive_expect_tx(fb, 3 * kStageTileBytes + ntok * 4);
        ptx::tma_load_3d(A(s.q[b]), &tmQ, fb, 0, st * ST, bh);
        ptx::tma_load_3d(A(s.k[b]), &tmK, fb, 0, st * ST, bh);
        ptx::tma_load_3d(A(s.v[b]), &tmV, fb, 0, st * ST, bh);
        ptx::bulk_load(A(s.eta[b]), eta_bh + st * ST, ntok * 4, fb);
    };
    if (tid == 0) {
        for (int i = 0; i < NSS; ++i) {
            ptx::mbar_init(A(&s.full[i]), 1);
            ptx::mbar_init(A(&s.empty[i]), 4);   // warps 0-3, after the stage's last output
        }
        for (int i = 0; i < 5; ++i) ptx::mbar_init(A(&s.mma[i]), 1);
        ptx::mbar_init(A(&s.x2r), kCompute);
        ptx::mbar_init(A(&s.g2r), 4);
        ptx::mbar_init(A(&s.g1r), kCompute);
        ptx::mbar_init(A(&s.xbr), kCompute);
        ptx::mbar_init(A(&s.prep), 1);
        ptx::mbar_init(A(&s.a2r), 1);
        ptx::mbar_init(A(&s.init), kCompute);
        ptx::mbar_init(A(&s.drain), 1);
        s.abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmZ);
    }
    if (warp == kCtl) {
        ptx::tmem_alloc(A(&s.tmem), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = s.tmem;

    auto wait = [&](unsigned long long *bar, uint32_t parity) -> bool {
        const uint32_t a = A(bar);
        if (ptx::mbar_try_wait(a, parity)) return true;
        return tmem_wait_slow(a, parity, p.wait_ns, &s.abort_flag, p.status);
    };

    if (warp == kCtl) {
        // ================================================================ control thread
        if (lane == 0) {
            const int nissue = p.withhold_loads ? 0 : p.NST;
            int issued = 0;
            for (; issued < min(NSS, nissue); ++issued) issue_stage(issued);
            const uint32_t w1t = A(s.w1t), w2t = A(s.w2t), w2 = A(s.w2), upd = A(s.upd), kte = A(s.kte);
            const uint32_t x2 = A(s.x2), xb2 = A(s.xb2), g2 = A(s.g2), a1 = A(s.a1), a2 = A(s.a2);
            bool ok = wait(&s.init, 0);
            for (int n = 0; n < N && ok; ++n) {
                const int st = n / TPS, slot = st % NSS, row0 = MB * (n % TPS);
                const uint32_t par = (uint32_t)(n & 1);
                if (!(ok = wait(&s.full[slot], (uint32_t)((st / NSS) & 1)))) break;
                ptx::tc_fence_after();
                // M1: Z1^T (keys | queries) = W1^T [K | Q]^T, K = 64 inputs in four K16 steps
                {
                    const uint32_t kt = A(s.k[slot]) + row0 * 128, qt = A(s.q[slot]) + row0 * 128;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = dsc(w1t + hf * 16384 + 32 * kk);
                            ptx::tc_mma(tmem + cZ1 + 32 * hf, ad, dsc(kt + 32 * kk), kI16, kk > 0);
                            ptx::tc_mma(tmem + cZ1 + 32 * hf + 16, ad, dsc(qt + 32 * kk), kI16, kk > 0);
                        }
                    ptx::tc_commit(A(&s.mma[0]));
                }
                // M2: Z2^T = W2^T X2^T, K = 256 hidden units in four 64-unit blocks
                if (!(ok = wait(&s.x2r, par))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::tc_mma(tmem + cZ2, dsc(w2t + j * 8192 + 32 * kk), dsc(x2 + j * 2048 + 32 * kk), kI16,
                                    (j | kk) > 0);
                ptx::tc_commit(A(&s.mma[1]));
                // M3: G1^T = W2 G2^T, K = 64 outputs
                if (!(ok = wait(&s.g2r, par))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::tc_mma(tmem + cG1 + 16 * hf, dsc(w2 + hf * 16384 + 32 * kk), dsc(g2 + 32 * kk), kI16,
                                    kk > 0);
                ptx::tc_commit(A(&s.mma[2]));
                // the previous stage's slot is read no more once its last output is written
                // (warps 0-3 do that before they publish this mini-batch's G2): refill it
                if (n % TPS == 0 && st >= 1 && st - 1 + NSS < nissue) {
                    const int old = st - 1;
                    if (!(ok = wait(&s.empty[old % NSS], (uint32_t)((old / NSS) & 1)))) break;
                    ptx::fence_proxy_async();
                    issue_stage(old + NSS);
                    issued = old + NSS + 1;
                }
                // M4: both updates and the query-side correction of the first layer (K = 16 tokens)
                if (!(ok = wait(&s.g1r, par))) break;
                if (!(ok = wait(&s.prep, par))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    ptx::tc_mma(tmem + cW1 + 64 * hf, dsc(upd + hf * 16384), dsc(kte), kI64, 1);
                    ptx::tc_mma(tmem + cW2 + 64 * hf, dsc(upd + hf * 16384 + 32), dsc(kte + 32), kI64, 1);
                    ptx::tc_mma(tmem + cZ1 + 32 * hf + 16, dsc(upd + hf * 16384), dsc(a1), kI16, 1);
                }
                ptx::tc_commit(A(&s.mma[3]));
                // M5: Zb2^T = W2^T Xb2^T + (-eta G2)^T A2^T
                if (!(ok = wait(&s.xbr, par))) break;
                if (!(ok = wait(&s.a2r, par))) break;
                ptx::tc_fence_after();
                {
                    const uint32_t dz = tmem + cZB2 + 16 * (n & 1);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            ptx::tc_mma(dz, dsc(w2t + j * 8192 + 32 * kk), dsc(xb2 + j * 2048 + 32 * kk), kI16,
                                        (j | kk) > 0);
                    ptx::tc_mma(dz, dsc(kte + 32), dsc(a2), kI16, 1);
                    ptx::tc_commit(A(&s.mma[4]));
                }
            }
            // every MMA issued has completed, every copy issued has landed
            ptx::tc_commit(A(&s.drain));
            ptx::mbar_wait_bounded(A(&s.drain), 0, kDrainNs);
            if (!ok)
                for (int st = max(0, issued - NSS); st < issued; ++st)
                    ptx::mbar_wait_bounded(A(&s.full[st % NSS]), (uint32_t)((st / NSS) & 1), kDrainNs);
        }
    } else {
        // ================================================================ compute warps
        const int hf = warp >> 2, q4 = warp & 3, hu = 128 * hf + 32 * q4 + lane;   // hidden unit
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);                      // lane quadrant
        const size_t init = p.init_per_batch ? (size_t)bh : (size_t)head;
        const float kf = p.ip ? 0.f : 1.f;

        // ---- state: fp32 W1^T row and W2 row of unit hu into TMEM, bf16 copies into shared memory
        float b1 = p.b1[init * DH + hu];
        {
            const float *W1 = p.W1 + init * D * DH, *W2 = p.W2 + init * DH * D;
            uint32_t r[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(W1[(size_t)(32 * half + j) * DH + hu]);
                ptx::tc_st32x32(tl + cW1 + 64 * hf + 32 * half, r);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[8 * c + e]);
                    *reinterpret_cast<uint4 *>(s.w1t + ptx::sw128(hu, 4 * half + c)) = pack8(v);
                }
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(W2[(size_t)hu * D + 32 * half + j]);
                ptx::tc_st32x32(tl + cW2 + 64 * hf + 32 * half, r);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[8 * c + e]);
                    *reinterpret_cast<uint4 *>(s.w2 + ptx::sw128(hu, 4 * half + c)) = pack8(v);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    *reinterpret_cast<uint16_t *>(s.w2t[hu >> 6] + el(32 * half + j, hu & 63)) =
                        bf16_bits(__uint_as_float(r[j]));
            }
            // K^T / (-eta G2)^T block: zero (rows 64-127 stay zero: the padded rows of M5's A)
            uint4 *kz = reinterpret_cast<uint4 *>(s.kte) + tid * 4;
#pragma unroll
            for (int i = 0; i < 4; ++i) kz[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        ptx::tc_wait_st();
        ptx::fence_proxy_async();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(A(&s.init));

        // ---- LayerNorm threads (warps 0-3): token lt of the mini-batch, outputs 8 part .. + 7
        const int lt = 4 * warp + (lane >> 3), part = lane & 7;
        float ga[8], be[8], g20[8], C1 = 0.f;
        float b2 = 0.f, b2prev = 0.f, pivot = 0.f;   // warps 0-1: output o = 32 warp + lane
        if (warp < 4) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                ga[e] = LN ? p.gamma[(size_t)head * D + 8 * part + e] : 1.f;
                be[e] = LN ? p.beta[(size_t)head * D + 8 * part + e] : 0.f;
                g20[e] = kf * ga[e] * ga[e];
            }
            if (LN)
                for (int o = 0; o < D; ++o) {
                    const float g = p.gamma[(size_t)head * D + o];
                    C1 = fmaf(kf * g, g, C1);
                }
            if (warp < 2) {
                b2 = p.b2[init * D + 32 * warp + lane];
                // LayerNorm pivot: the scan runs on b2 - mean(b2) (the LayerNorm and its backward
                // do not see a common shift of Z2) and adds it back at the end, so the one-pass
                // sums of z and z^2 stay free of cancellation when b2 carries a large offset
                if (LN) {
                    for (int o = 0; o < D; ++o) pivot += p.b2[init * D + o];
                    pivot *= 1.f / D;
                    b2 -= pivot;
                }
            }
        }

        // ---- helpers
        const int g = lane >> 2, c4 = lane & 3, mrow = lane & 7, mat = lane >> 3;
        // K^T and A1 = (q_t . k_s + 1) [s <= t] of mini-batch m (warp 5)
        auto prep = [&](int m) {
            const int st = m / TPS, slot = st % NSS, row0 = MB * (m % TPS);
            wait(&s.full[slot], (uint32_t)((st / NSS) & 1));
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = lane + 32 * hh;
                float v[16];
#pragma unroll
                for (int t = 0; t < MB; ++t)
                    v[t] = __bfloat162float(__ushort_as_bfloat16(
                        *reinterpret_cast<const uint16_t *>(s.k[slot] + el(row0 + t, i))));
                *reinterpret_cast<uint4 *>(s.kte + ptx::sw128(i, 0)) = pack8(v);
                *reinterpret_cast<uint4 *>(s.kte + ptx::sw128(i, 1)) = pack8(v + 8);
            }
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                uint32_t a[4], b[4];
                ptx::ldsm_x4(A(s.q[slot]) + ptx::sw128(row0 + (mat & 1) * 8 + mrow, 2 * qd + (mat >> 1)), a);
                ptx::ldsm_x4(A(s.k[slot]) + ptx::sw128(row0 + (mat >> 1) * 8 + mrow, 2 * qd + (mat & 1)), b);
                ptx::mma_bf16(acc[0], a, b[0], b[1]);
                ptx::mma_bf16(acc[1], a, b[2], b[3]);
            }
#pragma unroll
            for (int hs = 0; hs < 2; ++hs)
#pragma unroll
                for (int r2 = 0; r2 < 2; ++r2) {
                    const int t = g + 8 * r2, s0 = 8 * hs + 2 * c4;
                    const float v0 = s0 <= t ? acc[hs][2 * r2] + 1.f : 0.f;
                    const float v1 = s0 + 1 <= t ? acc[hs][2 * r2 + 1] + 1.f : 0.f;
                    *reinterpret_cast<uint32_t *>(s.a1 + el(t, s0)) = ptx::pack_bf16(v0, v1);
                }
            ptx::fence_proxy_async();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(A(&s.prep));
        };
        // A2 = (xb2_t . x2_s + 1) [s <= t] of mini-batch m (warps 6-7, one hidden half each)
        auto gram = [&](int m) {
            wait(&s.xbr, (uint32_t)(m & 1));
            const int kh = warp - kGramWarp;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float ac2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int qq = 0; qq < 8; ++qq) {
                const int q = 8 * kh + qq, blk = q >> 2, ch = 2 * (q & 3);
                uint32_t a[4], b[4];
                ptx::ldsm_x4(A(s.xb2[blk]) + ptx::sw128((mat & 1) * 8 + mrow, ch + (mat >> 1)), a);
                ptx::ldsm_x4(A(s.x2[blk]) + ptx::sw128((mat >> 1) * 8 + mrow, ch + (mat & 1)), b);
                float(*dst)[4] = (qq & 1) ? ac2 : acc;
                ptx::mma_bf16(dst[0], a, b[0], b[1]);
                ptx::mma_bf16(dst[1], a, b[2], b[3]);
            }
#pragma unroll
            for (int hs = 0; hs < 2; ++hs)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[hs][e] += ac2[hs][e];
            if (kh == 1) {
                float4 *dst = reinterpret_cast<float4 *>(s.gram[lane]);
                dst[0] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
                dst[1] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
            }
            ptx::named_bar(kBarGram, 64);
            if (kh == 0) {
                const float4 o0 = reinterpret_cast<const float4 *>(s.gram[lane])[0];
                const float4 o1 = reinterpret_cast<const float4 *>(s.gram[lane])[1];
                acc[0][0] += o0.x; acc[0][1] += o0.y; acc[0][2] += o0.z; acc[0][3] += o0.w;
                acc[1][0] += o1.x; acc[1][1] += o1.y; acc[1][2] += o1.z; acc[1][3] += o1.w;
#pragma unroll
                for (int hs = 0; hs < 2; ++hs)
#pragma unroll
                    for (int r2 = 0; r2 < 2; ++r2) {
                        const int t = g + 8 * r2, s0 = 8 * hs + 2 * c4;
                        const float v0 = s0 <= t ? acc[hs][2 * r2] + 1.f : 0.f;
                        const float v1 = s0 + 1 <= t ? acc[hs][2 * r2 + 1] + 1.f : 0.f;
                        *reinterpret_cast<uint32_t *>(s.a2 + el(t, s0)) = ptx::pack_bf16(v0, v1);
                    }
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(A(&s.a2r));
            }
        };
        // output of mini-batch m: Z = Q + LN(Zb2) (warps 0-3), TMA-stored from the staging tile
        auto ln_out = [&](int m) {
            const int st = m / TPS, slot = st % NSS, row0 = MB * (m % TPS);
            if (warp < 2) {
                uint32_t r[16];
                ptx::tc_ld32x16(tl + cZB2 + 16 * (m & 1), r);
                ptx::tc_wait_ld();
#pragma unroll
                for (int t = 0; t < MB; ++t) s.zb[t][32 * warp + lane] = __uint_as_float(r[t]) + b2prev;
            }
            if (tid == 0) ptx::bulk_wait_read<0>();   // the last store has read the staging tile
            ptx::named_bar(kBarLn, 128);
            float z[8], out[8];
            {
                const float4 z0 = *reinterpret_cast<const float4 *>(&s.zb[lt][8 * part]);
                const float4 z1 = *reinterpret_cast<const float4 *>(&s.zb[lt][8 * part + 4]);
                z[0] = z0.x; z[1] = z0.y; z[2] = z0.z; z[3] = z0.w;
                z[4] = z1.x; z[5] = z1.y; z[6] = z1.z; z[7] = z1.w;
            }
            if (LN) {
                float s1 = 0.f, s2 = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    s1 += z[e];
                    s2 = fmaf(z[e], z[e], s2);
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                    s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                }
                const float mu = s1 * (1.f / D);
                const float r = rsqrtf(fmaxf(s2 * (1.f / D) - mu * mu, 0.f) + p.eps);
                float qv[8];
                unpack8(*reinterpret_cast<const uint4 *>(s.q[slot] + ptx::sw128(row0 + lt, part)), qv);
#pragma unroll
                for (int e = 0; e < 8; ++e) out[e] = qv[e] + fmaf(ga[e] * (z[e] - mu), r, be[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) out[e] = z[e];
            }
            *reinterpret_cast<uint4 *>(s.zst + ptx::sw128(lt, part)) = pack8(out);
            ptx::fence_proxy_async();
            ptx::named_bar(kBarLn, 128);
            if (tid == 0) {
                ptx::tma_store_3d(&tmZ, A(s.zst), 0, m * MB, bh);
                ptx::bulk_commit();
            }
            if (m % TPS == TPS - 1) {   // the stage is read no more by warps 0-3
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(A(&s.empty[slot]));
            }
        };

        if (warp == kPrepWarp && N > 0) {
            wait(&s.init, 0);   // every warp has zeroed its part of the K^T block
            prep(0);
        }

        float dz[16];        // GELU'(Z1) of this unit's 16 tokens
        uint32_t w2p[32];    // the updated W2 row (bf16 pairs) for the W2^T columns
        for (int n = 0; n < N; ++n) {
            const int st = n / TPS, slot = st % NSS, row0 = MB * (n % TPS);
            const uint32_t par = (uint32_t)(n & 1);
            const float *et = s.eta[slot] + row0;
            // this thread reads the stage's eta (and warps 0-3 its K, V, Q rows): the copy landed
            wait(&s.full[slot], (uint32_t)((st / NSS) & 1));

            // ---- Z1 -> X2 = GELU(Z1) (a [t][h] column for M2, an [h][t] row for the W2 update)
            wait(&s.mma[0], par);
            ptx::tc_fence_after();
            {
                uint32_t r[16];
                ptx::tc_ld32x16(tl + cZ1 + 32 * hf, r);
                ptx::tc_wait_ld();
                float xv[16];
#pragma unroll
                for (int t = 0; t < MB; ++t) gelu_and_prime(__uint_as_float(r[t]) + b1, xv[t], dz[t]);
                unsigned char *xc = s.x2[hu >> 6];
#pragma unroll
                for (int t = 0; t < MB; ++t) *reinterpret_cast<uint16_t *>(xc + el(t, hu & 63)) = bf16_bits(xv[t]);
                *reinterpret_cast<uint4 *>(s.upd + ptx::sw128(hu, 2)) = pack8(xv);
                *reinterpret_cast<uint4 *>(s.upd + ptx::sw128(hu, 3)) = pack8(xv + 8);
            }
            ptx::fence_proxy_async();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(A(&s.x2r));

            if (warp < 4) {
                // ---- the previous mini-batch's output while M2 runs
                if (n > 0) ln_out(n - 1);
                // ---- Z2 -> G2 (LayerNorm backward), -eta G2, b2 -= eta^T G2
                wait(&s.mma[1], par);
                ptx::tc_fence_after();
                if (warp < 2) {
                    uint32_t r[16];
                    ptx::tc_ld32x16(tl + cZ2, r);
                    ptx::tc_wait_ld();
                    b2prev = b2;
#pragma unroll
                    for (int t = 0; t < MB; ++t) s.zb[t][32 * warp + lane] = __uint_as_float(r[t]) + b2;
                }
                ptx::named_bar(kBarLn, 128);
                float z[8], kv[8], vv[8], gm[8];
                {
                    const float4 z0 = *reinterpret_cast<const float4 *>(&s.zb[lt][8 * part]);
                    const float4 z1 = *reinterpret_cast<const float4 *>(&s.zb[lt][8 * part + 4]);
                    z[0] = z0.x; z[1] = z0.y; z[2] = z0.z; z[3] = z0.w;
                    z[4] = z1.x; z[5] = z1.y; z[6] = z1.z; z[7] = z1.w;
                }
                unpack8(*reinterpret_cast<const uint4 *>(s.v[slot] + ptx::sw128(row0 + lt, part)), vv);
                if (LN) {
                    unpack8(*reinterpret_cast<const uint4 *>(s.k[slot] + ptx::sw128(row0 + lt, part)), kv);
                    float gb[8], S[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        gb[e] = ga[e] * fmaf(kf, be[e] + kv[e], -vv[e]);
                        const float a = g20[e] * z[e];
                        S[0] += z[e];
                        S[1] = fmaf(z[e], z[e], S[1]);
                        S[2] += a;
                        S[3] = fmaf(a, z[e], S[3]);
                        S[4] = fmaf(gb[e], z[e], S[4]);
                        S[5] += gb[e];
                    }
#pragma unroll
                    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
                        for (int i = 0; i < 6; ++i) S[i] += __shfl_xor_sync(0xffffffffu, S[i], o);
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
                    for (int e = 0; e < 8; ++e)
                        gm[e] = fmaf(z[e] - mu, fmaf(co_a, g20[e], -co_b), fmaf(r, gb[e], -co_e));
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) gm[e] = fmaf(z[e], kf, -vv[e]);
                }
                *reinterpret_cast<uint4 *>(s.g2 + ptx::sw128(lt, part)) = pack8(gm);
                const float e_t = et[lt];
                float eg[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) eg[e] = -e_t * gm[e];
                *reinterpret_cast<float4 *>(&s.zb[lt][8 * part]) = make_float4(eg[0], eg[1], eg[2], eg[3]);
                *reinterpret_cast<float4 *>(&s.zb[lt][8 * part + 4]) = make_float4(eg[4], eg[5], eg[6], eg[7]);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    *reinterpret_cast<uint16_t *>(s.kte + el(8 * part + e, 16 + lt)) = bf16_bits(eg[e]);
                ptx::fence_proxy_async();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(A(&s.g2r));
                ptx::named_bar(kBarLn, 128);
                if (warp < 2) {
                    float acc = 0.f;
#pragma unroll
                    for (int t = 0; t < MB; ++t) acc += s.zb[t][32 * warp + lane];
                    b2 += acc;
                }
            }

            // ---- G1 = (G2 W2^T) . GELU'(Z1) -> -eta G1 as an [h][t] row; b1 -= eta^T G1 (after M4)
            float db1 = 0.f;
            wait(&s.mma[2], par);
            ptx::tc_fence_after();
            {
                uint32_t r[16];
                ptx::tc_ld32x16(tl + cG1 + 16 * hf, r);
                ptx::tc_wait_ld();
                float eg[16];
#pragma unroll
                for (int t = 0; t < MB; ++t) {
                    const float gv = __uint_as_float(r[t]) * dz[t], e = et[t];
                    eg[t] = -e * gv;
                    db1 = fmaf(e, gv, db1);
                }
                *reinterpret_cast<uint4 *>(s.upd + ptx::sw128(hu, 0)) = pack8(eg);
                *reinterpret_cast<uint4 *>(s.upd + ptx::sw128(hu, 1)) = pack8(eg + 8);
            }
            ptx::fence_proxy_async();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(A(&s.g1r));

            // ---- after M4: Xb2 = GELU(Zb1), and the bf16 copies of the updated W1^T and W2
            wait(&s.mma[3], par);
            ptx::tc_fence_after();
            {
                uint32_t r[32];
                ptx::tc_ld32x16(tl + cZ1 + 32 * hf + 16, r);
                ptx::tc_wait_ld();
                unsigned char *xc = s.xb2[hu >> 6];
#pragma unroll
                for (int t = 0; t < MB; ++t)
                    *reinterpret_cast<uint16_t *>(xc + el(t, hu & 63)) = bf16_bits(gelu(__uint_as_float(r[t]) + b1));
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    ptx::tc_ld32x32(tl + cW1 + 64 * hf + 32 * half, r);
                    ptx::tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[8 * c + e]);
                        *reinterpret_cast<uint4 *>(s.w1t + ptx::sw128(hu, 4 * half + c)) = pack8(v);
                    }
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    ptx::tc_ld32x32(tl + cW2 + 64 * hf + 32 * half, r);
                    ptx::tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[8 * c + e]);
                        const uint4 u = pack8(v);
                        *reinterpret_cast<uint4 *>(s.w2 + ptx::sw128(hu, 4 * half + c)) = u;
                        w2p[16 * half + 4 * c] = u.x;
                        w2p[16 * half + 4 * c + 1] = u.y;
                        w2p[16 * half + 4 * c + 2] = u.z;
                        w2p[16 * half + 4 * c + 3] = u.w;
                    }
                }
            }
            b1 -= db1;
            ptx::fence_proxy_async();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(A(&s.xbr));

            if (warp == kGramWarp || warp == kGramWarp + 1) gram(n);
            if (warp == kPrepWarp && n + 1 < N) prep(n + 1);

            // ---- W2^T for the next mini-batch, once M5 has read the old one
            wait(&s.mma[4], par);
            ptx::tc_fence_after();
            {
                unsigned char *wc = s.w2t[hu >> 6];
                const int col = hu & 63;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    *reinterpret_cast<uint16_t *>(wc + el(2 * j, col)) = (uint16_t)(w2p[j] & 0xffffu);
                    *reinterpret_cast<uint16_t *>(wc + el(2 * j + 1, col)) = (uint16_t)(w2p[j] >> 16);
                }
            }
        }
        if (warp < 4 && N > 0) ln_out(N - 1);

        // ---- final state
        {
            float *W1f = p.W1f + (size_t)bh * D * DH;
            float *W2f = p.W2f + (size_t)bh * DH * D;
            uint32_t r[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                ptx::tc_ld32x32(tl + cW1 + 64 * hf + 32 * half, r);
                ptx::tc_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) W1f[(size_t)(32 * half + j) * DH + hu] = __uint_as_float(r[j]);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                ptx::tc_ld32x32(tl + cW2 + 64 * hf + 32 * half, r);
                ptx::tc_wait_ld();
                float4 *dst = reinterpret_cast<float4 *>(W2f + (size_t)hu * D + 32 * half);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                         __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
            p.b1f[(size_t)bh * DH + hu] = b1;
            if (warp < 2) p.b2f[(size_t)bh * D + 32 * warp + lane] = b2 + pivot;
        }
        if (tid == 0) ptx::bulk_wait<0>();   // the output stores are complete
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kCtl) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool mlp_tmem_supported(const ttt_desc &d)
{
    return d.io_dtype == TTT_BF16 && d.d == D && d.d_hidden == DH && d.mini_batch == MB && d.weight_decay == 0.f;
}

cudaError_t launch_mlp_tmem(const MlpArgs &a)
{
    const ttt_desc &d = a.desc;
    const int BH = call_rows(d);
    CUtensorMap mq, mk, mv, mz;
    if (!make_bf16_tile_map(&mq, a.Q, d.L, BH, ST) || !make_bf16_tile_map(&mk, a.K, d.L, BH, ST) ||
        !make_bf16_tile_map(&mv, a.V, d.L, BH, ST) || !make_bf16_tile_map(&mz, a.Z, d.L, BH, MB))
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
    const size_t smem = sizeof(Smem) + 1024;
    auto kern = d.residual_ln ? mlp_tmem_kernel<true> : mlp_tmem_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<BH, kThreads, smem, a.stream>>>(mq, mk, mv, mz, p);
    return cudaGetLastError();
}

}  // namespace ttt
