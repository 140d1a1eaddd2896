// ttt_internal.h -- declarations shared by the host side of libttt.so
// (argument checks in ttt_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/ttt.h"

namespace ttt {

// Everything a launcher needs for one TTT-Linear call (pointers already checked).
struct LinearArgs {
    ttt_desc desc;
    const void *Q, *K, *V;
    const float *eta, *W0, *b0, *gamma, *beta;
    void *Z;
    float *W_final, *b_final;
    cudaStream_t stream;
    unsigned int *status;  // device-side failure flag (bounded waits)
};

struct MlpArgs {
    ttt_desc desc;  // desc.d_hidden already resolved (> 0)
    const void *Q, *K, *V;
    const float *eta, *W1_0, *b1_0, *W2_0, *b2_0, *gamma, *beta;
    void *Z;
    float *W1_f, *b1_f, *W2_f, *b2_f;
    cudaStream_t stream;
    unsigned int *status;
};

// One TTT-Linear decode call: tokens one at a time from the state (W, b), updated in place.
struct DecodeArgs {
    ttt_desc desc;  // desc.L = tokens of this call, desc.mini_batch = 1
    const void *Q, *K, *V;
    const float *eta;
    float *W, *b;
    const float *gamma, *beta;
    void *Z;
    cudaStream_t stream;
};

// One TTT-Linear backward call (pointers already checked; the workspace holds
// linear_bwd_workspace_bytes(desc) bytes, 256-byte aligned).
struct LinearBwdArgs {
    ttt_desc desc;
    const void *Q, *K, *V, *dZ;
    const float *eta, *W0, *b0, *gamma, *beta, *dW_final, *db_final;   // dW_final, db_final may be null (0)
    void *dQ, *dK, *dV;
    float *deta, *dW0, *db0, *dgamma, *dbeta;   // gamma, beta, dgamma, dbeta: residual LN only
    void *workspace;
    cudaStream_t stream;
};

// TTT-Linear backward (d <= 128, d % 4 == 0, b <= 64, shared memory permitting).  *_checkpoint_every returns the mini-batches per state checkpoint (0: the
// shape is not supported).
int linear_bwd_checkpoint_every(const ttt_desc &d);
size_t linear_bwd_workspace_bytes(const ttt_desc &d);
cudaError_t launch_linear_bwd(const LinearBwdArgs &a);

// One per-token learning-rate gate call: eta [B, H, L] from x [B, L, Dx] and theta [H, Dx].
struct GateArgs {
    int B, H, L, Dx;
    ttt_dtype x_dtype;
    float eta_base;
    const void *x;
    const float *theta;
    float *eta;
    cudaStream_t stream;
    unsigned int *status;
    int max_sms;   // > 0: at most this many SMs' worth of CTAs
};

// One input-projection call: Q, K, V [B, H, L, d] (bf16) from x [B, L, Dx] and the stacked
// projection matrices W [3 H d, Dx] (bf16).
struct ProjArgs {
    int B, H, L, Dx, d;
    const void *x, *W;
    __nv_bfloat16 *Q, *K, *V;
    cudaStream_t stream;
    unsigned int *status;
    int max_sms;   // > 0: at most this many SMs
};
bool qkv_proj_supported(int B, int H, int L, int Dx, int d);
cudaError_t launch_qkv_proj(const ProjArgs &a);

// Gate kernels: warp-MMA kernel for bf16 tokens (H <= 32, Dx % 16 == 0), FP32 otherwise.
bool gate_mma_supported(int H, int Dx, ttt_dtype x_dtype);
cudaError_t launch_eta_gate(const GateArgs &a);

// Generic kernels: one CTA per (batch, head), fp32 FFMA arithmetic, state in
// shared memory.  *_smem_bytes returns 0 when the shape does not fit.
size_t linear_generic_smem_bytes(const ttt_desc &d);
cudaError_t launch_linear_generic(const LinearArgs &a);
size_t mlp_generic_smem_bytes(const ttt_desc &d);
cudaError_t launch_mlp_generic(const MlpArgs &a);

// Column-split TTT-Linear kernel without the residual LayerNorm (fp32 FFMA, d <= 128,
// d % 4 == 0, b <= 64): each (batch, head) row runs on d / dc CTAs of dc output columns.
// linear_cols_dc returns dc, or 0 when the kernel is not used for the shape (LN, or too
// many rows for a split to pay).
int linear_cols_dc(const ttt_desc &d);
cudaError_t launch_linear_cols(const LinearArgs &a);

// Tensor-core TTT-Linear kernel (bf16 I/O, d = 64, b = 16).
bool linear_tc_supported(const ttt_desc &d);
cudaError_t launch_linear_tc(const LinearArgs &a);
// Chunked tensor-core TTT-Linear kernel without the residual LayerNorm (bf16 I/O, d = 64,
// b = 16, no weight decay): the state is carried across 64-token chunks.
bool linear_chunk_supported(const ttt_desc &d);
cudaError_t launch_linear_chunk(const LinearArgs &a);
// TMA map of a [rows][cols] bf16 matrix: boxes of box_rows rows x 64 columns, 128-byte swizzle.
bool make_bf16_2d_map(CUtensorMap *m, const void *base, unsigned long long rows, unsigned long long cols,
                      unsigned box_rows);
// TMA map of a [BH][L][64] bf16 tensor: boxes of `rows` tokens x 64 features, 128-byte swizzle.
bool make_bf16_tile_map(CUtensorMap *m, const void *base, int L, int BH, int rows);
// TTT-Linear decode kernel (d = 64, fp32 or bf16 I/O, FP32 arithmetic, one warp per head).
bool linear_decode_supported(const ttt_desc &d);
cudaError_t launch_linear_decode(const DecodeArgs &a);
// Tensor-core TTT-MLP kernel (bf16 I/O, d = 64, d_hidden = 256, b = 16).
bool mlp_tc_supported(const ttt_desc &d);
cudaError_t launch_mlp_tc(const MlpArgs &a);
// TTT-MLP with the hidden-width products on tcgen05 and W1^T, W2 resident in tensor memory
// (bf16 I/O, d = 64, d_hidden = 256, b = 16, no weight decay).
bool mlp_tmem_supported(const ttt_desc &d);
cudaError_t launch_mlp_tmem(const MlpArgs &a);
// Test hooks of the bounded waits (process-wide; see ttt.h), read by both fused kernels.
void set_wait_timeout_ns(long long ns);
void set_withhold_loads(int on);
long long wait_timeout_ns();
int withhold_loads();

// (batch, head) rows covered by one call, and the head index of its first row.  Row-indexed
// buffers start at the call's first row; head-indexed parameters are whole, and row i of the
// call uses head (bh_offset + i) mod H, i.e. (head_offset + i) mod H.
inline int call_rows(const ttt_desc &d) { return d.bh_count > 0 ? d.bh_count : d.B * d.H; }
inline int head_offset(const ttt_desc &d) { return d.bh_offset % d.H; }

// Error reports of ttt_linear_bwd_static (set ttt_last_error, return the status).
ttt_status fail_static_scratch(size_t need, size_t have);
ttt_status fail_cuda(const char *what, cudaError_t e);

// Device-side status word values.
enum : unsigned int { kStatusOk = 0u, kStatusTimeout = 1u };

}  // namespace ttt
