// ttt_gate.cu -- the per-token learning rate of the TTT layer (the learnable gate of the
// lryc.cn TTT article, section 2.2):
//   eta[b, h, t] = eta_base * sigmoid(theta[h] . x[b, t])
// for the layer's input tokens x [B, L, Dx] and one gate vector theta[h] [Dx] per head;
// eta [B, H, L] is the layout the scan kernels read.
//
// B300 design.  The gate is a skinny contraction ([B L, Dx] x [Dx, H], H <= 32) whose cost
// is reading x once: it is HBM-bound, so the kernel streams x at copy speed and keeps the
// arithmetic small.
//   * persistent CTAs (one per SM), 4 warps; 32-token tiles of x arrive as Dx / 64 TMA boxes
//     of 32 rows x 64 features (128-byte swizzle, so ldmatrix reads of eight rows hit eight
//     different bank groups) into a 2-4 deep shared-memory ring;
//   * theta is split once per CTA into bf16 hi + lo parts (theta = hi + lo to ~2^-16
//     relative), so bf16 tokens are contracted by warp MMAs (m16n8k16, fp32 accumulate)
//     with no precision lost beyond that split: logits = x . hi + x . lo;
//   * the epilogue applies eta_base / (1 + exp(-u)) and writes eta[b, h, t].
// The tensor-core form (eta_gate_tc_kernel) runs the contraction on tcgen05: 128-token tiles
// of x are the M side (TMA boxes of 128 rows x 64 features, 128-byte swizzle, in a 4-deep
// ring), theta hi and lo stacked as the N side (2 H rounded up to a multiple of 16, K-major
// in shared memory for the whole kernel), fp32 accumulators in tensor memory, double
// buffered so that the epilogue of one tile overlaps the MMAs of the next:
//   * warp 0: one thread issues the TMA loads (a slot is refilled once the MMAs that read it
//     have completed: tcgen05.commit on the slot's empty mbarrier);
//   * warp 1: allocates the tensor memory; one thread issues the 4 x (Dx / 64) MMAs of a tile
//     (M 128, N 2 H', K 16 each) and commits them to the accumulator's full mbarrier;
//   * warps 2-5: the epilogue, one TMEM lane quadrant each: tcgen05.ld of the token's 2 H'
//     logits (32x32b: thread = token), u = hi + lo, eta = eta_base / (1 + exp(-u)).
// The warp-MMA form stays for the shapes whose theta does not fit beside the ring; fp32
// tokens, widths that are no multiple of 64 or that no ring can hold take a plain FP32 kernel
// (one warp per token row).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kGateThreads = 128;
constexpr int TR = 32;                       // tokens per tile
constexpr size_t kSmemLimit = 227 * 1024;    // opt-in shared memory per CTA

struct GateParams {
    int rows, L, H, HP, Dx, DXP, nstage;
    float eta_base;
    const void *x;
    const float *theta;
    float *eta;
    unsigned int *status;
    long long wait_ns;
};

size_t mma_smem_bytes(int HP, int Dx, int nstage)
{
    // ring (1024-aligned), theta hi / lo (padded rows), mbarriers, alignment slack
    return 1024 + (size_t)nstage * TR * Dx * 2 + (size_t)2 * HP * (Dx + 8) * 2 + 64;
}

__device__ __forceinline__ void store_eta(const GateParams &p, int row, int h, float u)
{
    if (row < p.rows && h < p.H) {
        const int b = row / p.L, t = row - b * p.L;
        p.eta[((size_t)b * p.H + h) * p.L + t] = p.eta_base / (1.f + expf(-u));
    }
}

// x tiles of TR tokens arrive as Dx / 64 TMA boxes of TR rows x 64 features (128-byte swizzle,
// 4 KB each); theta hi / lo rows are padded by 16 bytes so ldmatrix reads of eight heads hit
// eight different bank groups.
__global__ void __launch_bounds__(kGateThreads, 1)
eta_gate_mma_kernel(const __grid_constant__ CUtensorMap tmX, GateParams p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // 1024-byte aligned
    const int nbox = p.Dx / 64;
    const uint32_t stage_bytes = (uint32_t)nbox * TR * 128;
    unsigned char *ring = smem;                                            // [nstage][nbox][TR][128 B]
    __nv_bfloat16 *th_hi = reinterpret_cast<__nv_bfloat16 *>(ring + (size_t)p.nstage * stage_bytes);
    __nv_bfloat16 *th_lo = th_hi + (size_t)p.HP * p.DXP;
    unsigned long long *full = reinterpret_cast<unsigned long long *>(th_lo + (size_t)p.HP * p.DXP);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (p.rows + TR - 1) / TR;

    if (tid == 0) {
        for (int s = 0; s < p.nstage; ++s) ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmX);
    }
    __syncthreads();

    // tile i of this CTA is global tile blockIdx.x + i * gridDim.x, in ring slot i % nstage
    auto issue = [&](int i) {   // one thread
        const int tile = blockIdx.x + i * gridDim.x;
        const int slot = i % p.nstage;
        const uint32_t bar = ptx::smem_addr(&full[slot]);
        ptx::mbar_arrive_expect_tx(bar, stage_bytes);
        const uint32_t dst = ptx::smem_addr(ring + (size_t)slot * stage_bytes);
        for (int kb = 0; kb < nbox; ++kb)
            ptx::tma_load_2d(dst + kb * TR * 128, &tmX, bar, kb * 64, tile * TR);
    };
    const int mine = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    int issued = min(p.nstage, mine);   // tiles handed to the copy engine (uniform in the CTA)
    if (tid == 0)
        for (int i = 0; i < issued; ++i) issue(i);

    // theta = hi + lo in bf16, rows H..HP-1 zero, while the first tiles are in flight;
    // float4 loads, eight in flight per thread
    {
        const int dx4 = p.Dx / 4, nvec = p.HP * dx4, nval = p.H * dx4;
        const float4 *th4 = reinterpret_cast<const float4 *>(p.theta);
        for (int base = tid; base < nvec; base += 8 * kGateThreads) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = base + u * kGateThreads;
                v[u] = i < nval ? th4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = base + u * kGateThreads;
                if (i < nvec) {
                    const int h = i / dx4, k = (i - h * dx4) * 4;
                    const float x4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                    uint32_t hi2[2], lo2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float a = x4[2 * e], b = x4[2 * e + 1];
                        hi2[e] = ptx::pack_bf16(a, b);
                        lo2[e] = ptx::pack_bf16(a - ptx::bf16_lo(hi2[e]), b - ptx::bf16_hi(hi2[e]));
                    }
                    *reinterpret_cast<uint2 *>(th_hi + h * p.DXP + k) = make_uint2(hi2[0], hi2[1]);
                    *reinterpret_cast<uint2 *>(th_lo + h * p.DXP + k) = make_uint2(lo2[0], lo2[1]);
                }
            }
        }
    }
    __syncthreads();

    const int g = lane >> 2, c = lane & 3, mrow = lane & 7;
    const int npairs = (TR / 16) * (p.HP / 8);   // (m-tile, n-tile) pairs of a TR x HP logit tile
    const uint32_t hi_base = ptx::smem_addr(th_hi), lo_base = ptx::smem_addr(th_lo);
    bool ok = true;
    for (int i = 0; i < mine; ++i) {
        const int slot = i % p.nstage, tile = blockIdx.x + i * gridDim.x;
        const uint32_t bar = ptx::smem_addr(&full[slot]);
        const uint32_t parity = (uint32_t)((i / p.nstage) & 1);
        bool landed = ptx::mbar_try_wait(bar, parity) || ptx::mbar_wait_bounded(bar, parity, p.wait_ns);
        // one verdict for the whole CTA, so that every thread takes the same branches below
        ok = __syncthreads_and(ok && landed) != 0;
        if (!ok) {
            if (tid == 0) atomicOr(p.status, kStatusTimeout);
            break;
        }
        const uint32_t xs = ptx::smem_addr(ring + (size_t)slot * stage_bytes);
        for (int pr = warp; pr < npairs; pr += 4) {
            const int mt = pr % (TR / 16), nt = pr / (TR / 16);
            // A: token row t of this lane's ldmatrix address (matrices: rows 0-7 / 8-15 x
            // k 0-7 / 8-15 of a 16-wide k-step); B: head row of theta hi (lanes 0-15) / lo
            const int t = mt * 16 + mrow + ((lane >> 3) & 1) * 8;
            const uint32_t a_row = xs + (uint32_t)(t * 128);
            const int a_half = lane >> 4;
            const uint32_t b_addr = ((lane >> 4) ? lo_base : hi_base) +
                                    (uint32_t)(((nt * 8 + mrow) * p.DXP + ((lane >> 3) & 1) * 8) * 2);
            float acc[4][4] = {};
            for (int kb = 0; kb < nbox; ++kb) {
                const uint32_t a_box = a_row + (uint32_t)(kb * TR * 128);
#pragma unroll
                for (int ks = 0; ks < 4; ks += 2) {
                    uint32_t a0[4], b0[4], a1[4], b1[4];
                    // 16-byte chunk (2 ks + a_half) of the 64-feature box row, swizzled
                    ptx::ldsm_x4(a_box + (uint32_t)((((2 * ks + a_half) ^ (t & 7))) << 4), a0);
                    ptx::ldsm_x4(b_addr + (uint32_t)((kb * 64 + ks * 16) * 2), b0);
                    ptx::ldsm_x4(a_box + (uint32_t)((((2 * ks + 2 + a_half) ^ (t & 7))) << 4), a1);
                    ptx::ldsm_x4(b_addr + (uint32_t)((kb * 64 + ks * 16 + 16) * 2), b1);
                    ptx::mma_bf16(acc[0], a0, b0[0], b0[1]);
                    ptx::mma_bf16(acc[1], a0, b0[2], b0[3]);
                    ptx::mma_bf16(acc[2], a1, b1[0], b1[1]);
                    ptx::mma_bf16(acc[3], a1, b1[2], b1[3]);
                }
            }
            float u4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) u4[k] = (acc[0][k] + acc[2][k]) + (acc[1][k] + acc[3][k]);
            const int r0 = tile * TR + mt * 16 + g, h0 = nt * 8 + 2 * c;
            store_eta(p, r0, h0, u4[0]);
            store_eta(p, r0, h0 + 1, u4[1]);
            store_eta(p, r0 + 8, h0, u4[2]);
            store_eta(p, r0 + 8, h0 + 1, u4[3]);
        }
        __syncthreads();   // every warp is done with the slot
        if (i + p.nstage < mine) {
            if (tid == 0) {
                ptx::fence_proxy_async();
                issue(i + p.nstage);
            }
            ++issued;
        }
    }
    // copies still in flight after a wait ran out land before the CTA exits
    if (!ok && tid == 0)
        for (int i = max(0, issued - p.nstage); i < issued; ++i)
            ptx::mbar_wait_bounded(ptx::smem_addr(&full[i % p.nstage]),
                                   (uint32_t)((i / p.nstage) & 1), 1000000000ll);
}

// ---------------------------------------------------------------- tcgen05 form
constexpr int TM = 128;                  // tokens per tile (the MMA's M)
constexpr int NSR_MAX = 4;               // ring stages of one 128 x 64 box each (at most)
constexpr int kTcThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kBoxBytes = TM * 128; // 16 KB

struct TcGateParams {
    int rows, L, H, HP, N, Dx, nkb, ncols, nst;
    float eta_base;
    const float *theta;
    float *eta;
    unsigned int *status;
    long long wait_ns;
};

size_t tc_smem_bytes(int N, int Dx, int nst)
{
    // ring + theta (1024-aligned regions), mbarriers + TMEM address + abort flag, slack
    return 1024 + (size_t)nst * kBoxBytes + (size_t)Dx * N * 2 + 256;
}

__global__ void __launch_bounds__(kTcThreads, 1)
eta_gate_tc_kernel(const __grid_constant__ CUtensorMap tmX, TcGateParams p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // 1024-byte aligned
    const int NSR = p.nst;
    unsigned char *ring = smem;                                            // [NSR][128 rows][128 B]
    unsigned char *thb = ring + NSR * kBoxBytes;                           // [nkb][N rows][128 B]
    unsigned long long *bars = reinterpret_cast<unsigned long long *>(thb + (size_t)p.Dx * p.N * 2);
    unsigned long long *full = bars, *empty = bars + NSR, *acc_full = bars + 2 * NSR,
                       *acc_empty = acc_full + 2, *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (p.rows + TM - 1) / TM;
    const int mine = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (tid == 0) {
        for (int i = 0; i < NSR; ++i) {
            ptx::mbar_init(ptx::smem_addr(&full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_addr(&acc_full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&acc_empty[i]), 4);   // one arrival per epilogue warp
        }
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmX);
    }
    // box kc (k-block kc % nkb of this CTA's tile kc / nkb) into ring slot kc % NSR
    auto load_box = [&](int kc) {
        const int tile = blockIdx.x + (kc / p.nkb) * gridDim.x, kb = kc % p.nkb, slot = kc % NSR;
        const uint32_t fb = ptx::smem_addr(&full[slot]);
        ptx::mbar_arrive_expect_tx(fb, kBoxBytes);
        ptx::tma_load_2d(ptx::smem_addr(ring + slot * kBoxBytes), &tmX, fb, kb * 64, tile * TM);
    };
    const int nbox = mine * p.nkb;
    const int first = min(NSR, nbox);   // boxes in flight before theta is converted
    if (tid == 0)
        for (int kc = 0; kc < first; ++kc) load_box(kc);
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), (uint32_t)p.ncols);
        ptx::tmem_relinquish();
    }
    // theta = hi + lo (bf16), rows 0..HP-1 hi, HP..2 HP-1 lo, zero past H; K-major with the
    // 128-byte swizzle: element (n, k) at kb N 128 + n 128 + ((k % 64 / 8) ^ (n % 8)) 16 + k % 8 * 2
    {
        // 16-byte chunks of the hi and lo rows; eight chunks' loads in flight per thread
        constexpr int kBatch = 16;
        const int units = p.N * (p.Dx / 8);
        for (int base = tid; base < units; base += kBatch * kTcThreads) {
            float4 va[kBatch], vb[kBatch];
#pragma unroll
            for (int r = 0; r < kBatch; ++r) {
                const int u = base + r * kTcThreads;
                const int n = u / (p.Dx / 8), k = (u - n * (p.Dx / 8)) * 8;
                const int h = n >= p.HP ? n - p.HP : n;
                if (u < units && h < p.H) {
                    va[r] = *reinterpret_cast<const float4 *>(p.theta + (size_t)h * p.Dx + k);
                    vb[r] = *reinterpret_cast<const float4 *>(p.theta + (size_t)h * p.Dx + k + 4);
                } else {
                    va[r] = vb[r] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int r = 0; r < kBatch; ++r) {
                const int u = base + r * kTcThreads;
                if (u >= units) break;
                const int n = u / (p.Dx / 8), k = (u - n * (p.Dx / 8)) * 8;
                const bool lo = n >= p.HP;
                const float v[8] = {va[r].x, va[r].y, va[r].z, va[r].w, vb[r].x, vb[r].y, vb[r].z, vb[r].w};
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t hi = ptx::pack_bf16(v[2 * e], v[2 * e + 1]);
                    w[e] = lo ? ptx::pack_bf16(v[2 * e] - ptx::bf16_lo(hi), v[2 * e + 1] - ptx::bf16_hi(hi)) : hi;
                }
                const int kb = k / 64, chunk = (k % 64) / 8;
                unsigned char *dst = thb + (size_t)kb * p.N * 128 + n * 128 + ((chunk ^ (n & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    ptx::fence_proxy_async();   // the generic-proxy theta writes, before the MMAs read them
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto give_up = [&]() {
        *(volatile int *)abort_flag = 1;
        atomicOr(p.status, kStatusTimeout);
    };
    auto wait = [&](unsigned long long *bar, uint32_t parity) -> bool {
        const uint32_t a = ptx::smem_addr(bar);
        if (ptx::mbar_try_wait(a, parity)) return true;
        if (*(volatile int *)abort_flag) return false;
        if (ptx::mbar_wait_bounded(a, parity, p.wait_ns)) return true;
        give_up();
        return false;
    };

    const uint32_t idesc = ptx::idesc_bf16_kk(TM, p.N);
    int loads = first;   // boxes handed to the copy engine (thread 0)
    if (warp == 0 && lane == 0) {
        // ---- TMA producer: the rest of the boxes, each once the MMAs have read its slot
        for (int kc = first; kc < nbox; ++kc) {
            if (!wait(&empty[kc % NSR], (uint32_t)(((kc / NSR) - 1) & 1))) break;
            load_box(kc);
            ++loads;
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        bool ok = true;
        for (int i = 0; i < mine && ok; ++i) {
            const int buf = i & 1;
            if (i >= 2 && !(ok = wait(&acc_empty[buf], (uint32_t)(((i / 2) - 1) & 1)))) break;
            ptx::tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(buf * p.N);
            for (int kb = 0; kb < p.nkb; ++kb) {
                const int kc = i * p.nkb + kb, slot = kc % NSR;
                if (!(ok = wait(&full[slot], (uint32_t)((kc / NSR) & 1)))) break;
                ptx::tc_fence_after();
                const uint32_t a0 = ptx::smem_addr(ring + slot * kBoxBytes);
                const uint32_t b0 = ptx::smem_addr(thb + (size_t)kb * p.N * 128);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    ptx::tc_mma(d, ptx::sdesc_sw128(a0 + 32 * kk), ptx::sdesc_sw128(b0 + 32 * kk), idesc,
                                (kb | kk) != 0);
                ptx::tc_commit(ptx::smem_addr(&empty[slot]));
            }
            if (ok) ptx::tc_commit(ptx::smem_addr(&acc_full[buf]));
        }
        // every MMA issued has completed before the tensor memory is freed
        ptx::tc_commit(ptx::smem_addr(drain));
        ptx::mbar_wait_bounded(ptx::smem_addr(drain), 0, 1000000000ll);
    } else if (warp >= 2) {
        // ---- epilogue: warp quadrant q reads TMEM lanes 32 q .. 32 q + 31 (token rows)
        const int q = warp & 3;
        for (int i = 0; i < mine; ++i) {
            const int buf = i & 1;
            if (!wait(&acc_full[buf], (uint32_t)((i / 2) & 1))) break;
            ptx::tc_fence_after();
            const int row = (blockIdx.x + i * gridDim.x) * TM + 32 * q + lane;
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * p.N);
            const int b = row / p.L, t = row - b * p.L;
            for (int c0 = 0; c0 < p.HP; c0 += 32) {   // 32 heads at a time: hi at c0, lo at HP + c0
                uint32_t hi[32], lo[32];
                ptx::tc_ld32x32(base + (uint32_t)c0, hi);
                ptx::tc_ld32x32(base + (uint32_t)(p.HP + c0), lo);
                ptx::tc_wait_ld();
                if (row < p.rows) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (c0 + j < p.H) {
                            const float u = __uint_as_float(hi[j]) + __uint_as_float(lo[j]);
                            p.eta[((size_t)b * p.H + c0 + j) * p.L + t] = p.eta_base / (1.f + expf(-u));
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&acc_empty[buf]));
        }
    }
    // copies still in flight after a wait ran out land before the CTA exits
    if (warp == 0 && lane == 0 && *(volatile int *)abort_flag)
        for (int kc = max(0, loads - NSR); kc < loads; ++kc)
            ptx::mbar_wait_bounded(ptx::smem_addr(&full[kc % NSR]), (uint32_t)((kc / NSR) & 1), 1000000000ll);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, (uint32_t)p.ncols);
}

// Plain FP32 gate: one warp per token row, every head.
template <bool BF16>
__global__ void __launch_bounds__(256) eta_gate_generic_kernel(GateParams p)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int row = warp; row < p.rows; row += nwarps) {
        for (int h = 0; h < p.H; ++h) {
            const float *th = p.theta + (size_t)h * p.Dx;
            float s = 0.f;
            for (int k = lane; k < p.Dx; k += 32) {
                float xv;
                if (BF16)
                    xv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.x)[(size_t)row * p.Dx + k]);
                else
                    xv = reinterpret_cast<const float *>(p.x)[(size_t)row * p.Dx + k];
                s = fmaf(xv, th[k], s);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) store_eta(p, row, h, s);
        }
    }
}

}  // namespace

// tcgen05 form: bf16 tokens, Dx a multiple of 64, N = 2 H' <= 256 (H' = H rounded up to 8,
// so that N is a multiple of 16) and theta fitting beside the ring.
int gate_tc_n(int H) { return 2 * ((H + 7) / 8 * 8); }
// tensor-memory columns: two accumulators of N columns, plus the 32-column reads of the
// epilogue that start inside the second one (at most N + HP + HP - 1 + 32 <= 2 N + 32)
int gate_tc_cols(int N)
{
    int c = 32;
    while (c < 2 * N + 32) c *= 2;
    return c;
}
bool gate_tc_supported(int H, int Dx, ttt_dtype x_dtype)
{
    if (x_dtype != TTT_BF16 || Dx % 64 != 0 || H < 1) return false;
    const int N = gate_tc_n(H);
    return N <= 224 && gate_tc_cols(N) <= 512 && tc_smem_bytes(N, Dx, 2) <= kSmemLimit;
}

bool gate_mma_supported(int H, int Dx, ttt_dtype x_dtype)
{
    if (x_dtype != TTT_BF16 || H > 32 || Dx % 64 != 0) return false;
    const int HP = H <= 16 ? 16 : 32;
    return mma_smem_bytes(HP, Dx, 2) <= kSmemLimit;
}

cudaError_t launch_eta_gate(const GateArgs &a)
{
    int dev = 0, sms = 148;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (a.max_sms > 0) sms = min(sms, a.max_sms);   // the caller leaves the other SMs to a scan
    GateParams p{};
    p.rows = a.B * a.L;
    p.L = a.L;
    p.H = a.H;
    p.Dx = a.Dx;
    p.eta_base = a.eta_base;
    p.x = a.x;
    p.theta = a.theta;
    p.eta = a.eta;
    p.status = a.status;
    p.wait_ns = wait_timeout_ns();
    if (gate_tc_supported(a.H, a.Dx, a.x_dtype)) {
        TcGateParams t{};
        t.rows = p.rows;
        t.L = a.L;
        t.H = a.H;
        t.N = gate_tc_n(a.H);
        t.HP = t.N / 2;
        t.Dx = a.Dx;
        t.nkb = a.Dx / 64;
        t.ncols = gate_tc_cols(t.N);
        t.nst = NSR_MAX;
        while (t.nst > 2 && tc_smem_bytes(t.N, a.Dx, t.nst) > kSmemLimit) --t.nst;
        t.eta_base = a.eta_base;
        t.theta = a.theta;
        t.eta = a.eta;
        t.status = a.status;
        t.wait_ns = p.wait_ns;
        const size_t smem = tc_smem_bytes(t.N, a.Dx, t.nst);
        const int ntiles = (p.rows + TM - 1) / TM;
        CUtensorMap mx;
        if (!make_bf16_2d_map(&mx, a.x, (unsigned long long)p.rows, (unsigned long long)a.Dx, TM))
            return cudaErrorInvalidValue;
        if ((e = cudaFuncSetAttribute(eta_gate_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem)) != cudaSuccess)
            return e;
        eta_gate_tc_kernel<<<min(ntiles, sms), kTcThreads, smem, a.stream>>>(mx, t);
    } else if (gate_mma_supported(a.H, a.Dx, a.x_dtype)) {
        p.HP = a.H <= 16 ? 16 : 32;
        p.DXP = a.Dx + 8;
        p.nstage = 4;
        while (p.nstage > 2 && mma_smem_bytes(p.HP, a.Dx, p.nstage) > kSmemLimit) --p.nstage;
        const size_t smem = mma_smem_bytes(p.HP, a.Dx, p.nstage);
        const int ntiles = (p.rows + TR - 1) / TR;
        CUtensorMap mx;
        if (!make_bf16_2d_map(&mx, a.x, (unsigned long long)p.rows, (unsigned long long)a.Dx, TR))
            return cudaErrorInvalidValue;
        if ((e = cudaFuncSetAttribute(eta_gate_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem)) != cudaSuccess)
            return e;
        eta_gate_mma_kernel<<<min(ntiles, sms), kGateThreads, smem, a.stream>>>(mx, p);
    } else {
        const int blocks = min((p.rows + 7) / 8, sms * 8);
        if (a.x_dtype == TTT_BF16)
            eta_gate_generic_kernel<true><<<blocks, 256, 0, a.stream>>>(p);
        else
            eta_gate_generic_kernel<false><<<blocks, 256, 0, a.stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace ttt
