// Chunkwise EFLA forward on CUDA cores in fp32, for the shapes and chunk lengths the
// tensor-core kernel does not cover: fp32 inputs, head sizes 32 / 64, chunk lengths 16 / 32
// (and 64).  Its buffers for a chunk of 64 tokens with d_k = d_v = 128 take 224 KB of
// shared memory, so 64 is its largest chunk length.
//
// Per chunk of C tokens with start state S ("Exact Flow Linear Attention" (gist.science),
// Metodologia 3; "Error-Free Linear Attention is a Free Lunch" (howistudyai), Step 4):
//   alpha_t = -expm1(-beta_t lambda_t) / lambda_t,  lambda_t = ||k_t||^2   (beta_t at lambda_t = 0)
//   A       = strictly-lower( alpha_t k_t . k_s )
//   U       = (I + A)^{-1} diag(alpha) (V - K S)      (forward substitution, row by row)
//   O       = Q S + (Q K^T o M) U                     (M lower-triangular including the diagonal)
//   S      <- S + K^T U
// which is the token recurrence S_t = S_{t-1} + k_t u_t^T, u_t = alpha_t (v_t - S_{t-1}^T k_t),
// o_t = S_t^T q_t, unrolled over the chunk.  The triangular system is solved by forward
// substitution instead of forming (I + A)^{-1}: the same solution, with fewer operations on CUDA
// cores.
//
// One CTA of 256 threads per (sequence, head); K, Q, U (V, then R = V - K S, then the rank-1
// writes), O, the chunk's A and P = Q K^T o M, and S are fp32 in shared memory.
#include "internal.cuh"

namespace efla {
namespace {

constexpr int THREADS = 256;

// Shared memory of one CTA in floats: K, Q [C][dk], U, O [C][dv], A, P [C][C], S [dk][dv].
__host__ __device__ constexpr size_t simt_smem_floats(int C, int dk, int dv) {
    return (size_t)2 * C * dk + (size_t)2 * C * dv + (size_t)2 * C * C + (size_t)dk * dv;
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(THREADS, 1) chunk_simt_kernel(FwdArgs a) {
    extern __shared__ float smem[];
    const int C = a.chunk, dk = a.dk, dv = a.dv;
    float *Ks = smem, *Qs = Ks + C * dk, *Us = Qs + C * dk, *Os = Us + C * dv;
    float *As = Os + C * dv, *Ps = As + C * C, *Ss = Ps + C * C;
    __shared__ float alpha_s[128];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = blockIdx.x / a.H, h = blockIdx.x % a.H;
    long b, bos, eos;
    if (a.cu_seqlens) {
        b = 0;
        bos = a.cu_seqlens[n];
        eos = a.cu_seqlens[n + 1];
        if (bos < 0 || eos < bos || eos > a.T) {  // malformed bounds: flag and touch nothing
            if (tid == 0) atomicExch(a.status, (int)EFLA_ERR_INVALID_ARG);
            return;
        }
    } else {
        b = n;
        bos = 0;
        eos = a.T;
    }
    const TIn *q = static_cast<const TIn *>(a.q);
    const TIn *k = static_cast<const TIn *>(a.k);
    const TIn *v = static_cast<const TIn *>(a.v);
    TOut *o = static_cast<TOut *>(a.o);
    const size_t sbase = ((size_t)n * a.H + h) * dk * dv;

    for (int e = tid; e < dk * dv; e += THREADS) Ss[e] = a.S0 ? a.S0[sbase + e] : 0.f;

    const int nch = (int)((eos - bos + C - 1) / C);
    for (long t0 = bos; t0 < eos; t0 += C) {
        const int valid = (int)min((long)C, eos - t0);
        __syncthreads();  // the previous chunk is done with every buffer
        if (a.states) {  // the chunk's start state (chunked backward)
            float *dst = a.states + ((size_t)blockIdx.x * nch + (t0 - bos) / C) * dk * dv;
            for (int e = tid; e < dk * dv; e += THREADS) dst[e] = Ss[e];
        }
        // inputs of the chunk (rows past its end are zero)
        for (int e = tid; e < C * dk; e += THREADS) {
            const int t = e / dk, i = e % dk;
            const size_t row = ((size_t)b * a.T + (size_t)(t0 + t)) * a.H + h;
            Ks[e] = t < valid ? to_f32(k[row * dk + i]) : 0.f;
            Qs[e] = t < valid ? to_f32(q[row * dk + i]) : 0.f;
        }
        for (int e = tid; e < C * dv; e += THREADS) {
            const int t = e / dv, j = e % dv;
            const size_t row = ((size_t)b * a.T + (size_t)(t0 + t)) * a.H + h;
            Us[e] = t < valid ? to_f32(v[row * dv + j]) : 0.f;
        }
        __syncthreads();
        // lambda_t and alpha_t, one warp per row
        for (int t = warp; t < C; t += THREADS / 32) {
            float lam = 0.f;
            for (int i = lane; i < dk; i += 32) lam = fmaf(Ks[t * dk + i], Ks[t * dk + i], lam);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
            if (lane == 0) {
                const size_t row = ((size_t)b * a.T + (size_t)(t0 + t)) * a.H + h;
                alpha_s[t] = t < valid ? efla_alpha(a.beta[row], lam, a.euler) : 0.f;
            }
        }
        __syncthreads();
        // A[t][s] = alpha_t k_t.k_s (s < t), P[t][s] = q_t.k_s (s <= t)
        for (int e = tid; e < C * C; e += THREADS) {
            const int t = e / C, s = e % C;
            float kk = 0.f, qk = 0.f;
            if (s <= t) {
                for (int ii = 0; ii < dk; ++ii) {
                    const int i = (ii + s) & (dk - 1);  // rotated start: neighbouring threads hit distinct banks
                    const float ks = Ks[s * dk + i];
                    kk = fmaf(Ks[t * dk + i], ks, kk);
                    qk = fmaf(Qs[t * dk + i], ks, qk);
                }
            }
            As[e] = s < t ? alpha_s[t] * kk : 0.f;
            Ps[e] = s <= t ? qk : 0.f;
        }
        // R = V - K S into U, and O = Q S (S is the chunk's start state)
        for (int e = tid; e < C * dv; e += THREADS) {
            const int t = e / dv, j = e % dv;
            float x = 0.f, y = 0.f;
            for (int i = 0; i < dk; ++i) {
                const float sij = Ss[i * dv + j];
                x = fmaf(Ks[t * dk + i], sij, x);
                y = fmaf(Qs[t * dk + i], sij, y);
            }
            Us[e] -= x;
            Os[e] = y;
        }
        __syncthreads();
        // forward substitution, one thread per column: u_t = alpha_t R_t - sum_{s<t} A[t][s] u_s
        for (int j = tid; j < dv; j += THREADS) {
            for (int t = 0; t < valid; ++t) {
                float acc = alpha_s[t] * Us[t * dv + j];
                for (int s = 0; s < t; ++s) acc = fmaf(-As[t * C + s], Us[s * dv + j], acc);
                Us[t * dv + j] = acc;
            }
        }
        __syncthreads();
        // O += P U, written out; S += K^T U
        for (int e = tid; e < C * dv; e += THREADS) {
            const int t = e / dv, j = e % dv;
            if (t >= valid) continue;
            float y = Os[e];
            for (int s = 0; s <= t; ++s) y = fmaf(Ps[t * C + s], Us[s * dv + j], y);
            const size_t row = ((size_t)b * a.T + (size_t)(t0 + t)) * a.H + h;
            if (o) o[row * dv + j] = from_f32<TOut>(y);
        }
        for (int e = tid; e < dk * dv; e += THREADS) {
            const int i = e / dv, j = e % dv;
            float sv = Ss[e];
            for (int t = 0; t < valid; ++t) sv = fmaf(Ks[t * dk + i], Us[t * dv + j], sv);
            Ss[e] = sv;
        }
    }
    __syncthreads();
    if (a.S_T)
        for (int e = tid; e < dk * dv; e += THREADS) a.S_T[sbase + e] = Ss[e];
}

template <typename TIn, typename TOut>
cudaError_t launch_typed(const FwdArgs &a) {
    const size_t bytes = simt_smem_floats(a.chunk, a.dk, a.dv) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<TIn, TOut>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    chunk_simt_kernel<TIn, TOut><<<(unsigned)((long)a.N * a.H), THREADS, bytes, a.stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_simt(const FwdArgs &a) {
    if (a.N == 0) return cudaSuccess;
    const bool in_bf16 = a.in_dtype == EFLA_BF16, out_bf16 = a.o_dtype == EFLA_BF16;
    if (in_bf16)
        return out_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(a) : launch_typed<__nv_bfloat16, float>(a);
    return out_bf16 ? launch_typed<float, __nv_bfloat16>(a) : launch_typed<float, float>(a);
}

}  // namespace efla
