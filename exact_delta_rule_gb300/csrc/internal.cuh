// Internal declarations shared by the translation units of libefla.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "efla.h"

namespace efla {

// Library-owned device status word (EFLA_OK or EFLA_ERR_DEVICE_TIMEOUT).
// Defined in efla_api.cu; kernels in other units reach it through a pointer
// obtained with cudaGetSymbolAddress, passed as a kernel argument.
int *device_status_ptr();
// Bound on the chunk kernel's inter-role waits, in ns (efla_debug_set_wait_limit_ns; 2 s by default).
unsigned long long wait_limit_ns();
// Test hook (efla_debug_set_stall): bit STALL_CHUNK, STALL_BWD_STATE or STALL_BWD_GRAD makes
// that tensor-core kernel's MMA thread first wait on a barrier that nothing completes, so the
// wait runs out and the kernel takes its abort path.
enum { STALL_CHUNK = 1, STALL_BWD_STATE = 2, STALL_BWD_GRAD = 4 };
int debug_stall();

struct FwdArgs {
    const void *q, *k, *v;
    const float *beta;
    const float *S0;
    const int32_t *cu_seqlens;
    void *o;
    float *S_T;
    int B, T, H, dk, dv, N;
    efla_dtype in_dtype, o_dtype;
    int chunk;
    cudaStream_t stream;
    int *status;  // library device status word
    int euler;    // 1: delta-rule gate alpha = beta instead of the exact gate
    // Split sequences (tensor-core path only): segments of seg_len tokens, G per row of
    // [B, T]; maps != nullptr selects the segment-map launch, else s_in holds the
    // segments' start states (see the chunk kernel).
    int seg_len = 0, G = 0;
    const float *s_in = nullptr;
    float *maps = nullptr;
    // Chunked backward: the state at the start of every chunk, [N, H, nchunks] x dk x dv x 4 bytes
    // (rows of [B, T] only; o may then be nullptr): fp32 row-major from the CUDA-core chunk
    // kernel, bf16 hi/lo operand tiles (tc::put_col_split_tile) from the tensor-core one.
    float *states = nullptr;
    // With states, the tensor-core chunk kernel also writes every chunk's T'' (bf16 hi/lo operand
    // tile, [64][64] each, 128-byte swizzle: 16 KB a chunk) here, or nowhere if nullptr.
    uint8_t *tpp = nullptr;
};

struct DecodeArgs {
    const void *q, *k, *v;
    const float *beta;
    float *S;
    void *o;
    int B, H, dk, dv;
    efla_dtype in_dtype, o_dtype;
    cudaStream_t stream;
    int euler;
    int m = 1;  // tokens per sequence (multi-token decode)
};

struct PrepArgs {
    const void *k, *v;
    const float *beta;
    float *lam, *alpha;
    void *ak, *av;
    long long n;
    int dk, dv;
    efla_dtype dtype;
    int euler;
    cudaStream_t stream;
};

// Launchers return a cudaError_t from the launch (cudaSuccess if nothing launched).
cudaError_t launch_recurrent(const FwdArgs &a);
cudaError_t launch_decode(const DecodeArgs &a);
cudaError_t launch_decode_tokens(const DecodeArgs &a);
// tcgen05 multi-token decode: bf16 q, k, v, d_k = d_v = 128 (decode_tc.cu).
cudaError_t launch_decode_tokens_tc(const DecodeArgs &a, const char **why);
// Backward pass (bwd.cu): gradients of the forward over whole rows of [B, T].
struct BwdArgs {
    const void *q, *k, *v;
    const float *beta, *S0, *dO, *dST;
    float *dq, *dk, *dv, *dbeta, *dS0;
    int B, T, H, dk_dim, dv_dim;
    efla_dtype in_dtype;
    cudaStream_t stream;
    int euler;
};
cudaError_t launch_bwd(const BwdArgs &a);
// Chunked backward (bwd_chunk.cu), chunk 64, rows of [B, T]: the state gradients at the ends of
// the chunks, then every chunk's gradients in parallel from `states` (the forward's chunk-start
// states, filled first by a forward launch with FwdArgs::states).  dse: [B, H, nchunks, dk, dv].
cudaError_t launch_bwd_chunked(const BwdArgs &a, const float *states, float *dse);
// The same state pass on the tensor cores (bwd_tc.cu): bf16 q, k, d_k = d_v = 128, T > 0, after
// the forward with chunk-start states and T'' tiles (tpp);
// do_split is scratch for dO as bf16 hi and lo (2 x B*T*H*128 bf16); it also writes G of every
// token into g_out (B*T*H*128 fp32), dR into dv, -dR as bf16 hi and lo into dr_split (like
// do_split), and dse as bf16 hi/lo operand tiles, for launch_bwd_grad_tc.
cudaError_t launch_bwd_state_tc(const BwdArgs &a, float *dse, const uint8_t *tpp, void *do_split, float *g_out,
                                void *dr_split, const char **why);
// Per-chunk gradients on the tensor cores (bwd_grad_tc.cu) after launch_bwd_state_tc: reads the
// forward's chunk-start states and T'' tiles (FwdArgs::states, ::tpp), dse (all as bf16 hi/lo
// operand tiles), do_split, G (g) and dr_split; writes dq, dk, dbeta.
cudaError_t launch_bwd_grad_tc(const BwdArgs &a, const float *states, const float *dse, const uint8_t *tpp,
                               const void *do_split, const float *g, const void *dr_split, const char **why);
// [B, T, H, 128] bf16 tensor map of the backward kernels: box 64 features x 1 head x 64 tokens
// x 1, 128-byte swizzle (bwd_tc.cu).
bool bwd_row_map(CUtensorMap *m, const void *ptr, int B, int T, int H);

// Start states of the segments of split sequences from the segment maps (scan.cu).
cudaError_t launch_scan_combine(const float *S0, const float *maps, float *s_in, int B, int G, int H,
                                cudaStream_t stream);
cudaError_t launch_prep(const PrepArgs &a);
// tcgen05 chunk kernel: bf16 inputs, d_k = d_v = 128, chunk 64.
cudaError_t launch_chunk_tc(const FwdArgs &a, const char **why);
// Chunkwise forward on CUDA cores (fp32), every supported head size, chunk 16, 32 or 64.
cudaError_t launch_chunk_simt(const FwdArgs &a);

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// d alpha / d beta and d alpha / d lambda of alpha = f(beta, lambda) (fp32; a series in
// z = beta*lambda where the difference form cancels).
__device__ __forceinline__ void gate_grad(float beta, float lam, int euler, float &dfdb, float &dfdl) {
    if (euler) {
        dfdb = 1.f;
        dfdl = 0.f;
        return;
    }
    const float z = beta * lam;
    if (lam > 0.f && fabsf(z) >= 0.1f) {
        const float e = expf(-z);
        const float f = -expm1f(-z) / lam;
        dfdb = e;
        dfdl = (beta * e - f) / lam;
    } else {
        dfdb = lam > 0.f ? expf(-z) : 1.f;
        dfdl = beta * beta * (-0.5f + z * (1.f / 3.f + z * (-1.f / 8.f + z * (1.f / 30.f - z * (1.f / 144.f)))));
    }
}

// alpha = (1 - e^{-beta*lam}) / lam, evaluated as -expm1(-beta*lam)/lam; beta at lam == 0.
// With `euler` the delta-rule gate alpha = beta.
__device__ __forceinline__ float efla_alpha(float beta, float lam, int euler) {
    if (euler) return beta;
    return lam > 0.f ? -expm1f(-beta * lam) / lam : beta;
}

}  // namespace efla
