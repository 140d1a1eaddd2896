// ttt_gate.cu -- the per-token learning rate of the TTT layer (the learnable gate of the
// lryc.cn TTT article, section 2.2):
//   eta[b, h, t] = eta_base * sigmoid(theta[h] . x[b, t])
// for the layer's input tokens x [B, L, Dx] and one gate vector theta[h] [Dx] per head;
// eta [B, H, L] is the layout the scan kernels read.
//
// B300 design.  The gate is a skinny contraction ([B L, Dx] x [Dx, H], H <= 32) whose cost
// is reading x once: it is HBM-bound, so the kernel streams x at copy speed and keeps the
// arithmetic small.
//   * persistent CTAs (one per SM), 4 warps; 32-token tiles of x arrive by per-row bulk
//     copies (cp.async.bulk, one per token row, issued by the 32 lanes of warp 0) into a
//     2-3 deep shared-memory ring; each row is padded by 16 bytes so that ldmatrix reads of
//     eight consecutive rows hit eight different bank groups;
//   * theta is split once per CTA into bf16 hi + lo parts (theta = hi + lo to ~2^-16
//     relative), so bf16 tokens are contracted by warp MMAs (m16n8k16, fp32 accumulate)
//     with no precision lost beyond that split: logits = x . hi + x . lo;
//   * the epilogue applies eta_base / (1 + exp(-u)) and writes eta[b, h, t].
// fp32 tokens, more than 32 heads or widths the ring cannot hold take a plain FP32 kernel
// (one warp per token row).
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

size_t mma_smem_bytes(int HP, int DXP, int nstage)
{
    return 1024 + (size_t)2 * HP * DXP * 2 + (size_t)nstage * TR * DXP * 2;
}

__device__ __forceinline__ void store_eta(const GateParams &p, int row, int h, float u)
{
    if (row < p.rows && h < p.H) {
        const int b = row / p.L, t = row - b * p.L;
        p.eta[((size_t)b * p.H + h) * p.L + t] = p.eta_base / (1.f + expf(-u));
    }
}

__global__ void __launch_bounds__(kGateThreads, 1) eta_gate_mma_kernel(GateParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned long long *full = reinterpret_cast<unsigned long long *>(smem);   // [nstage]
    __nv_bfloat16 *th_hi = reinterpret_cast<__nv_bfloat16 *>(smem + 1024);
    __nv_bfloat16 *th_lo = th_hi + (size_t)p.HP * p.DXP;
    __nv_bfloat16 *ring = th_lo + (size_t)p.HP * p.DXP;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (p.rows + TR - 1) / TR;
    const int stage_elems = TR * p.DXP;

    if (tid == 0) {
        for (int s = 0; s < p.nstage; ++s) ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();

    // tile i of this CTA is global tile blockIdx.x + i * gridDim.x, in ring slot i % nstage
    auto issue = [&](int i) {   // warp 0 only
        const int tile = blockIdx.x + i * gridDim.x;
        const int slot = i % p.nstage;
        const int nrows = min(TR, p.rows - tile * TR);
        const uint32_t bar = ptx::smem_addr(&full[slot]);
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar, (uint32_t)(nrows * p.Dx * 2));
        __syncwarp();
        if (lane < nrows) {
            const __nv_bfloat16 *src =
                reinterpret_cast<const __nv_bfloat16 *>(p.x) + (size_t)(tile * TR + lane) * p.Dx;
            ptx::bulk_load(ptx::smem_addr(ring + (size_t)slot * stage_elems + lane * p.DXP), src,
                           (uint32_t)(p.Dx * 2), bar);
        }
    };
    const int mine = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    int issued = min(p.nstage, mine);   // tiles handed to the copy engine (uniform in the CTA)
    if (warp == 0)
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

    const int g = lane >> 2, c = lane & 3;
    const int npairs = 2 * (p.HP / 8);   // (m-tile, n-tile) pairs of a 32 x HP logit tile
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
        {
            const uint32_t xs = ptx::smem_addr(ring + (size_t)slot * stage_elems);
            for (int pr = warp; pr < npairs; pr += 4) {
                const int mt = pr & 1, nt = pr >> 1;
                // A rows (tokens) of this lane's ldmatrix address; B rows (heads)
                const uint32_t a_addr =
                    xs + (uint32_t)(((mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * p.DXP + (lane >> 4) * 8) * 2);
                const uint32_t b_addr = ((lane >> 4) ? lo_base : hi_base) +
                                        (uint32_t)(((nt * 8 + (lane & 7)) * p.DXP + ((lane >> 3) & 1) * 8) * 2);
                // four independent accumulator chains: (hi, lo) x (even, odd k-step)
                float acc[4][4] = {};
                for (int k = 0; k < p.Dx; k += 32) {
                    uint32_t a0[4], b0[4], a1[4], b1[4];
                    ptx::ldsm_x4(a_addr + k * 2, a0);
                    ptx::ldsm_x4(b_addr + k * 2, b0);
                    ptx::mma_bf16(acc[0], a0, b0[0], b0[1]);
                    ptx::mma_bf16(acc[1], a0, b0[2], b0[3]);
                    if (k + 16 < p.Dx) {
                        ptx::ldsm_x4(a_addr + (k + 16) * 2, a1);
                        ptx::ldsm_x4(b_addr + (k + 16) * 2, b1);
                        ptx::mma_bf16(acc[2], a1, b1[0], b1[1]);
                        ptx::mma_bf16(acc[3], a1, b1[2], b1[3]);
                    }
                }
                float u4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) u4[i] = (acc[0][i] + acc[2][i]) + (acc[1][i] + acc[3][i]);
                const int r0 = tile * TR + mt * 16 + g, h0 = nt * 8 + 2 * c;
                store_eta(p, r0, h0, u4[0]);
                store_eta(p, r0, h0 + 1, u4[1]);
                store_eta(p, r0 + 8, h0, u4[2]);
                store_eta(p, r0 + 8, h0 + 1, u4[3]);
            }
        }
        __syncthreads();   // every warp is done with the slot
        if (i + p.nstage < mine) {
            if (warp == 0) issue(i + p.nstage);
            ++issued;
        }
    }
    // copies still in flight after a wait ran out land before the CTA exits
    if (!ok && tid == 0)
        for (int i = max(0, issued - p.nstage); i < issued; ++i)
            ptx::mbar_wait_bounded(ptx::smem_addr(&full[i % p.nstage]),
                                   (uint32_t)((i / p.nstage) & 1), 1000000000ll);
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

bool gate_mma_supported(int H, int Dx, ttt_dtype x_dtype)
{
    if (x_dtype != TTT_BF16 || H > 32 || Dx % 16 != 0) return false;
    const int HP = H <= 16 ? 16 : 32, DXP = Dx + 8;
    return mma_smem_bytes(HP, DXP, 2) <= kSmemLimit;
}

cudaError_t launch_eta_gate(const GateArgs &a)
{
    int dev = 0, sms = 148;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
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
    if (gate_mma_supported(a.H, a.Dx, a.x_dtype)) {
        p.HP = a.H <= 16 ? 16 : 32;
        p.DXP = a.Dx + 8;
        p.nstage = 3;
        while (p.nstage > 2 && mma_smem_bytes(p.HP, p.DXP, p.nstage) > kSmemLimit) --p.nstage;
        const size_t smem = mma_smem_bytes(p.HP, p.DXP, p.nstage);
        const int ntiles = (p.rows + TR - 1) / TR;
        if ((e = cudaFuncSetAttribute(eta_gate_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem)) != cudaSuccess)
            return e;
        eta_gate_mma_kernel<<<min(ntiles, sms), kGateThreads, smem, a.stream>>>(p);
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
