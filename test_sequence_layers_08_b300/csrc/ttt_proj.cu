// ttt_proj.cu -- the TTT layer's input projections (the lryc.cn TTT article, section 2.2: the
// views XQ = x theta_Q, XK = x theta_K, XV = x theta_V of the layer's input tokens, one d-wide
// slice per head) in the layout the scan kernels read:
//   Q[b, h, t, j] = sum_i x[b, t, i] W[0 H d + h d + j, i]      (W: the three projection
//   K[b, h, t, j] = sum_i x[b, t, i] W[1 H d + h d + j, i]       matrices stacked, [3 H d, Dx],
//   V[b, h, t, j] = sum_i x[b, t, i] W[2 H d + h d + j, i]       each row one output unit)
// bf16 inputs, fp32 accumulation, bf16 outputs.
//
// B300 design.  A dense contraction ([B L, Dx] x [Dx, 3 H d]; 155 GFLOP for 4 x 8192 tokens
// of 768 features into 3 x 16 heads of 64) on tcgen05, persistent CTAs (one per SM):
//   * tiles of 128 tokens x 256 output units; the K dimension (Dx) streams in 64-feature
//     chunks: a TMA box of x (128 rows x 64 features, 16 KB) and one of W (256 rows x 64
//     features, 32 KB), 128-byte swizzle, into a 4-deep ring; both operands K-major;
//   * warp 0: one thread issues the TMA loads, refilling a slot once the MMAs that read it
//     have completed (tcgen05.commit on the slot's empty mbarrier);
//   * warp 1: allocates tensor memory (two fp32 accumulators of 256 columns: the epilogue of
//     one tile overlaps the MMAs of the next); one thread issues M128 N256 K16 MMAs, four per
//     chunk, and commits each tile to its accumulator's full mbarrier;
//   * warps 2-5: the epilogue, one tensor-memory lane quadrant each (thread = token row):
//     tcgen05.ld of 64 columns (one head), bf16 conversion into a 32-row x 128-byte staging
//     tile (128-byte swizzle, so the 32 row writes hit distinct banks), and one TMA store of
//     the tile: the warp's 32 tokens of one head are 4 KB of contiguous Q, K or V [B, H, L, d]
//     rows.  Two staging tiles per warp, so converting one head overlaps the store of the
//     last.  Per-thread 16-byte stores of the same rows (32 lines touched by every warp store)
//     took a third of the kernel's time; they remain only for 32-token groups that cross a
//     sequence boundary or run past the last token;
//   * CTAs run in clusters of two on the same 256 output units and neighbouring 128-token
//     tiles: rank 0 multicasts each W chunk into both CTAs' rings (the source is this GPU's
//     own memory), each CTA loads its own x chunk, and each CTA's MMA completion is committed
//     to the empty mbarriers of both, so a slot is refilled only once both have read it.  W,
//     the larger operand stream, crosses L2 half as often as with single CTAs;
//   * pair tiles are ordered output-units fastest, so the clusters working at the same time
//     share x through L2 (x leaves HBM about once; W stays in L2).
// Every mbarrier wait is bounded; a wait that runs out sets the failure flag and the kernel
// finishes without waiting again.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int TM = 128;                       // tokens per tile (MMA M)
constexpr int TN = 256;                       // output units per tile (MMA N)
constexpr int NST = 4;                        // ring stages
constexpr int kThreads = 192;                 // 6 warps
constexpr uint32_t kABytes = TM * 128;        // x box: 128 rows x 64 bf16
constexpr uint32_t kBBytes = TN * 128;        // W box: 256 rows x 64 bf16
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kOutBytes = 32 * 128;      // one epilogue warp's staging tile: 32 tokens x 64 bf16
constexpr int kTmemCols = 2 * TN;             // two accumulators
constexpr int kCluster = 2;                   // CTAs per cluster (W shared by multicast)

struct ProjParams {
    int M, L, H, d, Dx, nkb, ntn, npair;      // M = B L tokens; ntn = (3 H d) / TN; npair tiles of 2 x 128 tokens
    __nv_bfloat16 *Q, *K, *V;
    unsigned int *status;
    long long wait_ns;
};

size_t proj_smem_bytes() { return 1024 + (size_t)NST * kStageBytes + 4 * 2 * kOutBytes + 256; }

__global__ void __launch_bounds__(kThreads, 1)
qkv_proj_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, ProjParams p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // 1024-byte aligned
    unsigned char *ring = smem;                                            // [NST][A | B]
    unsigned char *outst = ring + (size_t)NST * kStageBytes;               // [4 warps][2][32 x 128 B]
    unsigned long long *bars = reinterpret_cast<unsigned long long *>(outst + 4 * 2 * kOutBytes);
    unsigned long long *full = bars, *empty = bars + NST, *acc_full = bars + 2 * NST, *acc_empty = acc_full + 2,
                       *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)ptx::cluster_rank(), cl = blockIdx.x / kCluster, ncl = gridDim.x / kCluster;
    // pair tile q of this cluster: 256 output units nt, tokens 256 mp .. + 255, this CTA's half
    // 128 (2 mp + rank) (past M: zero-filled loads, no stores); the same sequence in both CTAs
    const int mine = cl < p.npair ? (p.npair - 1 - cl) / ncl + 1 : 0;
    const int nchunk = mine * p.nkb;
    auto tile_of = [&](int i, int &mt, int &nt) {
        const int q = cl + i * ncl, mp = q / p.ntn;
        nt = q - mp * p.ntn;
        mt = 2 * mp + rank;
    };

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            ptx::mbar_init(ptx::smem_addr(&full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[i]), kCluster);   // both CTAs' MMAs have read it
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_addr(&acc_full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&acc_empty[i]), 4);   // one arrival per epilogue warp
        }
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmX);
        ptx::prefetch_tmap(&tmW);
    }
    // chunk kc: k-block kc % nkb of this CTA's tile kc / nkb, into ring slot kc % NST: its own
    // x box, and (rank 0) the W box for both CTAs; each CTA's full mbarrier expects both
    auto load_chunk = [&](int kc) {
        const int kb = kc % p.nkb, slot = kc % NST;
        int mt, nt;
        tile_of(kc / p.nkb, mt, nt);
        const uint32_t fb = ptx::smem_addr(&full[slot]);
        unsigned char *st = ring + (size_t)slot * kStageBytes;
        ptx::mbar_arrive_expect_tx(fb, kStageBytes);
        ptx::tma_load_2d(ptx::smem_addr(st), &tmX, fb, kb * 64, mt * TM);
        if (rank == 0) ptx::tma_load_2d_mc(ptx::smem_addr(st + kABytes), &tmW, fb, kb * 64, nt * TN, 0x3);
    };
    // the peer's mbarriers exist before any multicast copy or commit reaches them
    ptx::cluster_sync();
    const int first = min(NST, nchunk);
    if (tid == 0)
        for (int kc = 0; kc < first; ++kc) load_chunk(kc);
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), (uint32_t)kTmemCols);
        ptx::tmem_relinquish();
    }
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

    const uint32_t idesc = ptx::idesc_bf16_kk(TM, TN);
    int loads = first;   // chunks handed to the copy engine (thread 0)
    if (warp == 0 && lane == 0) {
        // ---- TMA producer: the rest of the chunks, each once the MMAs have read its slot
        for (int kc = first; kc < nchunk; ++kc) {
            if (!wait(&empty[kc % NST], (uint32_t)(((kc / NST) - 1) & 1))) break;
            load_chunk(kc);
            ++loads;
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        bool ok = true;
        for (int i = 0; i < mine && ok; ++i) {
            const int buf = i & 1;
            if (i >= 2 && !(ok = wait(&acc_empty[buf], (uint32_t)(((i / 2) - 1) & 1)))) break;
            ptx::tc_fence_after();
            const uint32_t dacc = tmem + (uint32_t)(buf * TN);
            for (int kb = 0; kb < p.nkb; ++kb) {
                const int kc = i * p.nkb + kb, slot = kc % NST;
                if (!(ok = wait(&full[slot], (uint32_t)((kc / NST) & 1)))) break;
                ptx::tc_fence_after();
                const uint32_t a0 = ptx::smem_addr(ring + (size_t)slot * kStageBytes);
                const uint32_t b0 = a0 + kABytes;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    ptx::tc_mma(dacc, ptx::sdesc_sw128(a0 + 32 * kk), ptx::sdesc_sw128(b0 + 32 * kk), idesc,
                                (kb | kk) != 0);
                ptx::tc_commit_mc(ptx::smem_addr(&empty[slot]), 0x3);   // in both CTAs
            }
            if (ok) ptx::tc_commit(ptx::smem_addr(&acc_full[buf]));
        }
        // every MMA issued has completed before the tensor memory is freed
        ptx::tc_commit(ptx::smem_addr(drain));
        ptx::mbar_wait_bounded(ptx::smem_addr(drain), 0, 1000000000ll);
    } else if (warp >= 2) {
        // ---- epilogue: warp quadrant q reads TMEM lanes 32 q .. 32 q + 31 (token rows)
        const int q = warp & 3;
        const int Hd = p.H * p.d;
        unsigned char *stage = outst + (size_t)q * 2 * kOutBytes;
        int nst = 0;   // staged stores issued by this warp (lane 0)
        for (int i = 0; i < mine; ++i) {
            const int buf = i & 1;
            if (!wait(&acc_full[buf], (uint32_t)((i / 2) & 1))) break;
            ptx::tc_fence_after();
            int mt, nt;
            tile_of(i, mt, nt);
            const int row0 = mt * TM + 32 * q, row = row0 + lane;
            const int b = row / p.L, t = row - b * p.L;
            // the warp's 32 tokens are one contiguous run of rows of each head's output
            const bool staged = row0 + 31 < p.M && row0 / p.L == (row0 + 31) / p.L;
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * TN);
#pragma unroll 1
            for (int c0 = 0; c0 < TN; c0 += 64) {   // one head's 64 units at a time
                uint32_t v0[32], v1[32];
                ptx::tc_ld32x32(base + (uint32_t)c0, v0);
                ptx::tc_ld32x32(base + (uint32_t)(c0 + 32), v1);
                ptx::tc_wait_ld();
                const int n = nt * TN + c0;                      // first unit of the head
                const int which = n / Hd, h = (n - which * Hd) / p.d;
                if (staged) {
                    unsigned char *tile = stage + (size_t)(nst & 1) * kOutBytes;
                    // the store issued two heads ago has finished reading this tile
                    if (lane == 0) ptx::bulk_wait_read<1>();
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(tile + ptx::sw128(lane, c)) =
                            make_uint4(ptx::pack_bf16(__uint_as_float(v0[8 * c]), __uint_as_float(v0[8 * c + 1])),
                                       ptx::pack_bf16(__uint_as_float(v0[8 * c + 2]), __uint_as_float(v0[8 * c + 3])),
                                       ptx::pack_bf16(__uint_as_float(v0[8 * c + 4]), __uint_as_float(v0[8 * c + 5])),
                                       ptx::pack_bf16(__uint_as_float(v0[8 * c + 6]), __uint_as_float(v0[8 * c + 7])));
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(tile + ptx::sw128(lane, 4 + c)) =
                            make_uint4(ptx::pack_bf16(__uint_as_float(v1[8 * c]), __uint_as_float(v1[8 * c + 1])),
                                       ptx::pack_bf16(__uint_as_float(v1[8 * c + 2]), __uint_as_float(v1[8 * c + 3])),
                                       ptx::pack_bf16(__uint_as_float(v1[8 * c + 4]), __uint_as_float(v1[8 * c + 5])),
                                       ptx::pack_bf16(__uint_as_float(v1[8 * c + 6]), __uint_as_float(v1[8 * c + 7])));
                    ptx::fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        const CUtensorMap *tm = which == 0 ? &tmQ : which == 1 ? &tmK : &tmV;
                        ptx::tma_store_3d(tm, ptx::smem_addr(tile), 0, row0 - b * p.L, b * p.H + h);
                        ptx::bulk_commit();
                    }
                    ++nst;
                } else if (row < p.M) {
                    __nv_bfloat16 *dst = (which == 0 ? p.Q : which == 1 ? p.K : p.V) +
                                         (((size_t)b * p.H + h) * p.L + t) * p.d;
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        d4[c] = make_uint4(ptx::pack_bf16(__uint_as_float(v0[8 * c]), __uint_as_float(v0[8 * c + 1])),
                                           ptx::pack_bf16(__uint_as_float(v0[8 * c + 2]), __uint_as_float(v0[8 * c + 3])),
                                           ptx::pack_bf16(__uint_as_float(v0[8 * c + 4]), __uint_as_float(v0[8 * c + 5])),
                                           ptx::pack_bf16(__uint_as_float(v0[8 * c + 6]), __uint_as_float(v0[8 * c + 7])));
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        d4[4 + c] = make_uint4(ptx::pack_bf16(__uint_as_float(v1[8 * c]), __uint_as_float(v1[8 * c + 1])),
                                               ptx::pack_bf16(__uint_as_float(v1[8 * c + 2]), __uint_as_float(v1[8 * c + 3])),
                                               ptx::pack_bf16(__uint_as_float(v1[8 * c + 4]), __uint_as_float(v1[8 * c + 5])),
                                               ptx::pack_bf16(__uint_as_float(v1[8 * c + 6]), __uint_as_float(v1[8 * c + 7])));
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&acc_empty[buf]));
        }
        // the staged stores have read shared memory and written Q, K, V before the CTA exits
        if (lane == 0) ptx::bulk_wait<0>();
    }
    // copies still in flight after a wait ran out land before the CTA exits
    if (warp == 0 && lane == 0 && *(volatile int *)abort_flag)
        for (int kc = max(0, loads - NST); kc < loads; ++kc)
            ptx::mbar_wait_bounded(ptx::smem_addr(&full[kc % NST]), (uint32_t)((kc / NST) & 1), 1000000000ll);
    ptx::tc_fence_before();
    __syncthreads();
    // no CTA leaves while its peer may still commit to its mbarriers or copy into its ring
    ptx::cluster_sync();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, (uint32_t)kTmemCols);
}

}  // namespace

bool qkv_proj_supported(int B, int H, int L, int Dx, int d)
{
    const long long M = (long long)B * L, N = 3LL * H * d;
    return d == 64 && Dx % 64 == 0 && Dx > 0 && N % TN == 0 && M > 0 && M <= 0x7fffffffLL && B > 0 && L > 0;
}

cudaError_t launch_qkv_proj(const ProjArgs &a)
{
    const int M = a.B * a.L, N = 3 * a.H * a.d;
    CUtensorMap mx, mw, mq, mk, mv;
    if (!make_bf16_2d_map(&mx, a.x, (unsigned long long)M, (unsigned long long)a.Dx, TM) ||
        !make_bf16_2d_map(&mw, a.W, (unsigned long long)N, (unsigned long long)a.Dx, TN) ||
        // output boxes of 32 tokens of one head (sequences shorter than that are never staged)
        !make_bf16_tile_map(&mq, a.Q, a.L, a.B * a.H, min(32, a.L)) ||
        !make_bf16_tile_map(&mk, a.K, a.L, a.B * a.H, min(32, a.L)) ||
        !make_bf16_tile_map(&mv, a.V, a.L, a.B * a.H, min(32, a.L)))
        return cudaErrorInvalidValue;
    ProjParams p;
    p.M = M;
    p.L = a.L;
    p.H = a.H;
    p.d = a.d;
    p.Dx = a.Dx;
    p.nkb = a.Dx / 64;
    p.ntn = N / TN;
    p.npair = ((M + 2 * TM - 1) / (2 * TM)) * p.ntn;
    p.Q = a.Q;
    p.K = a.K;
    p.V = a.V;
    p.status = a.status;
    p.wait_ns = wait_timeout_ns();
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int cap = a.max_sms > 0 ? max(1, min(a.max_sms, sms) / kCluster) : sms;   // clusters
    const size_t smem = proj_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(qkv_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // persistent: as many clusters as can be resident at once (the two CTAs of a cluster sit in
    // one GPC, so this can be fewer than half the SMs), never more than there are pair tiles
    static std::atomic<int> resident[64];   // per device; 0 = not yet asked
    int active = dev >= 0 && dev < 64 ? resident[dev].load(std::memory_order_relaxed) : 0;
    if (active < 1) {
        cfg.gridDim = dim3(sms);
        if (cudaOccupancyMaxActiveClusters(&active, qkv_proj_kernel, &cfg) != cudaSuccess || active < 1) {
            (void)cudaGetLastError();
            active = sms / kCluster;
        }
        if (dev >= 0 && dev < 64) resident[dev].store(active, std::memory_order_relaxed);
    }
    cfg.gridDim = dim3(kCluster * min(min(p.npair, active), cap));
    return cudaLaunchKernelEx(&cfg, qkv_proj_kernel, mx, mw, mq, mk, mv, p);
}

}  // namespace ttt
