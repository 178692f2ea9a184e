// CUDA-core (fp32 FFMA) kernels: the single-token decode step and the
// token-by-token forward.
//
// Both evaluate, per head, one application per token of
//   lambda = ||k||^2,  alpha = -expm1(-beta*lambda)/lambda (beta at lambda = 0),
//   S <- (I - alpha k k^T) S + alpha k v^T,  o = S^T q with the updated S
// ["Exact Flow Linear Attention" (gist.science), Metodologia 3;
//  "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-3]
// in the single-pass form
//   x = S^T k, y = S^T q, u = alpha (v - x), o = y + (q.k) u, S += k u^T,
// which reads the old S once, because S_new^T q = S^T q + u (k.q).
#include "internal.cuh"

namespace efla {
namespace {

// ---------------------------------------------------------------------------
// Decode: one CTA of 256 threads per (b, h).  S[b,h] (d_k x d_v fp32, d_v
// contiguous) is read once into registers with 16-byte loads and written once.
// Thread layout: CG = DV/4 column groups of 4 floats (lanes along d_v, so each
// row is one contiguous warp access), RG = 256/CG row groups, each thread
// holding DK/RG rows of its 4 columns.
// ---------------------------------------------------------------------------
template <int DK, int DV, typename TIn, typename TOut>
__global__ void __launch_bounds__(256) decode_kernel(const TIn *__restrict__ q,
                                                     const TIn *__restrict__ k,
                                                     const TIn *__restrict__ v,
                                                     const float *__restrict__ beta,
                                                     float *__restrict__ S,
                                                     TOut *__restrict__ o, int euler) {
    constexpr int CG = DV / 4;
    constexpr int RG = 256 / CG;
    constexpr int ROWS = DK / RG;
    static_assert(ROWS >= 1 && DK % RG == 0, "unsupported decode shape");

    __shared__ float ks[DK], qs[DK];
    __shared__ float red_x[RG][DV], red_y[RG][DV];
    __shared__ float us[DV];
    __shared__ float scal[2];

    const int unit = blockIdx.x;  // b * H + h
    const int tid = threadIdx.x;
    const int cg = tid % CG, rg = tid / CG;

    float4 *Su = reinterpret_cast<float4 *>(S + (size_t)unit * DK * DV);
    float4 reg[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) reg[r] = Su[(size_t)(rg + r * RG) * CG + cg];

    if (tid < DK) {
        ks[tid] = to_f32(k[(size_t)unit * DK + tid]);
        qs[tid] = to_f32(q[(size_t)unit * DK + tid]);
    }
    __syncthreads();
    if (tid < 32) {
        float lam = 0.f, qk = 0.f;
        for (int i = tid; i < DK; i += 32) {
            lam = fmaf(ks[i], ks[i], lam);
            qk = fmaf(qs[i], ks[i], qk);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            lam += __shfl_xor_sync(0xffffffffu, lam, off);
            qk += __shfl_xor_sync(0xffffffffu, qk, off);
        }
        if (tid == 0) {
            scal[0] = efla_alpha(beta[unit], lam, euler);
            scal[1] = qk;
        }
    }

    float px[4] = {0.f, 0.f, 0.f, 0.f}, py[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const float ki = ks[rg + r * RG], qi = qs[rg + r * RG];
        const float s4[4] = {reg[r].x, reg[r].y, reg[r].z, reg[r].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            px[c] = fmaf(ki, s4[c], px[c]);
            py[c] = fmaf(qi, s4[c], py[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        red_x[rg][cg * 4 + c] = px[c];
        red_y[rg][cg * 4 + c] = py[c];
    }
    __syncthreads();
    if (tid < DV) {
        float x = 0.f, y = 0.f;
#pragma unroll 8
        for (int r = 0; r < RG; ++r) {
            x += red_x[r][tid];
            y += red_y[r][tid];
        }
        const float a = scal[0], qk = scal[1];
        const float u = a * (to_f32(v[(size_t)unit * DV + tid]) - x);
        us[tid] = u;
        o[(size_t)unit * DV + tid] = from_f32<TOut>(fmaf(qk, u, y));
    }
    __syncthreads();
    const float u0 = us[cg * 4 + 0], u1 = us[cg * 4 + 1], u2 = us[cg * 4 + 2], u3 = us[cg * 4 + 3];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const float ki = ks[rg + r * RG];
        float4 s = reg[r];
        s.x = fmaf(ki, u0, s.x);
        s.y = fmaf(ki, u1, s.y);
        s.z = fmaf(ki, u2, s.z);
        s.w = fmaf(ki, u3, s.w);
        Su[(size_t)(rg + r * RG) * CG + cg] = s;
    }
}

// ---------------------------------------------------------------------------
// Token-by-token forward: one warp per (sequence, head, 32-column slab of d_v).
// Lane j owns column j of S (DK fp32 registers), so S^T k and S^T q need no
// cross-lane reduction; k and q of the current token are staged in shared
// memory and read as broadcasts.
// ---------------------------------------------------------------------------
template <int DK, typename TIn, typename TOut>
__global__ void __launch_bounds__(128) recurrent_kernel(FwdArgs a) {
    __shared__ float ks_all[4][DK], qs_all[4][DK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slabs = a.dv / 32;
    const long unit = (long)blockIdx.x * 4 + warp;
    if (unit >= (long)a.N * a.H * slabs) return;
    const int slab = (int)(unit % slabs);
    const int h = (int)((unit / slabs) % a.H);
    const int n = (int)(unit / ((long)slabs * a.H));
    const int j = slab * 32 + lane;
    float *ks = ks_all[warp], *qs = qs_all[warp];

    long t0, t1, b;
    if (a.cu_seqlens) {
        b = 0;
        t0 = a.cu_seqlens[n];
        t1 = a.cu_seqlens[n + 1];
        if (t0 < 0 || t1 < t0 || t1 > a.T) {  // malformed bounds: flag and touch nothing
            if (lane == 0) atomicExch(a.status, (int)EFLA_ERR_INVALID_ARG);
            return;
        }
    } else {
        b = n;
        t0 = 0;
        t1 = a.T;
    }
    const TIn *q = static_cast<const TIn *>(a.q);
    const TIn *k = static_cast<const TIn *>(a.k);
    const TIn *v = static_cast<const TIn *>(a.v);
    TOut *o = static_cast<TOut *>(a.o);
    const size_t sbase = ((size_t)n * a.H + h) * DK * a.dv;

    float s[DK];
#pragma unroll
    for (int i = 0; i < DK; ++i) s[i] = a.S0 ? a.S0[sbase + (size_t)i * a.dv + j] : 0.f;

    for (long t = t0; t < t1; ++t) {
        const size_t row = ((size_t)b * a.T + t) * a.H + h;
        float lam = 0.f, qk = 0.f;
#pragma unroll
        for (int i = lane; i < DK; i += 32) {
            const float kv = to_f32(k[row * DK + i]), qv = to_f32(q[row * DK + i]);
            ks[i] = kv;
            qs[i] = qv;
            lam = fmaf(kv, kv, lam);
            qk = fmaf(qv, kv, qk);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            lam += __shfl_xor_sync(0xffffffffu, lam, off);
            qk += __shfl_xor_sync(0xffffffffu, qk, off);
        }
        __syncwarp();
        const float alpha = efla_alpha(a.beta[row], lam, a.euler);
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int i = 0; i < DK; ++i) {
            x = fmaf(ks[i], s[i], x);
            y = fmaf(qs[i], s[i], y);
        }
        const float u = alpha * (to_f32(v[row * a.dv + j]) - x);
        o[row * a.dv + j] = from_f32<TOut>(fmaf(qk, u, y));
#pragma unroll
        for (int i = 0; i < DK; ++i) s[i] = fmaf(ks[i], u, s[i]);
        __syncwarp();
    }
    if (a.S_T) {
#pragma unroll
        for (int i = 0; i < DK; ++i) a.S_T[sbase + (size_t)i * a.dv + j] = s[i];
    }
}

template <int DK, int DV, typename TIn, typename TOut>
cudaError_t decode_launch(const DecodeArgs &a) {
    decode_kernel<DK, DV, TIn, TOut><<<a.B * a.H, 256, 0, a.stream>>>(
        static_cast<const TIn *>(a.q), static_cast<const TIn *>(a.k),
        static_cast<const TIn *>(a.v), a.beta, a.S, static_cast<TOut *>(a.o), a.euler);
    return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t decode_dispatch_types(const DecodeArgs &a) {
    const bool ib = a.in_dtype == EFLA_BF16, ob = a.o_dtype == EFLA_BF16;
    if (ib && ob) return decode_launch<DK, DV, __nv_bfloat16, __nv_bfloat16>(a);
    if (ib) return decode_launch<DK, DV, __nv_bfloat16, float>(a);
    if (ob) return decode_launch<DK, DV, float, __nv_bfloat16>(a);
    return decode_launch<DK, DV, float, float>(a);
}

template <int DK>
cudaError_t decode_dispatch_dv(const DecodeArgs &a) {
    switch (a.dv) {
        case 32: return decode_dispatch_types<DK, 32>(a);
        case 64: return decode_dispatch_types<DK, 64>(a);
        default: return decode_dispatch_types<DK, 128>(a);
    }
}

template <int DK, typename TIn, typename TOut>
cudaError_t recurrent_launch(const FwdArgs &a) {
    const long units = (long)a.N * a.H * (a.dv / 32);
    const long blocks = (units + 3) / 4;
    recurrent_kernel<DK, TIn, TOut><<<(unsigned)blocks, 128, 0, a.stream>>>(a);
    return cudaGetLastError();
}

template <int DK>
cudaError_t recurrent_dispatch_types(const FwdArgs &a) {
    const bool ib = a.in_dtype == EFLA_BF16, ob = a.o_dtype == EFLA_BF16;
    if (ib && ob) return recurrent_launch<DK, __nv_bfloat16, __nv_bfloat16>(a);
    if (ib) return recurrent_launch<DK, __nv_bfloat16, float>(a);
    if (ob) return recurrent_launch<DK, float, __nv_bfloat16>(a);
    return recurrent_launch<DK, float, float>(a);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a) {
    if (a.B == 0) return cudaSuccess;
    switch (a.dk) {
        case 32: return decode_dispatch_dv<32>(a);
        case 64: return decode_dispatch_dv<64>(a);
        default: return decode_dispatch_dv<128>(a);
    }
}

cudaError_t launch_recurrent(const FwdArgs &a) {
    if (a.N == 0) return cudaSuccess;
    switch (a.dk) {
        case 32: return recurrent_dispatch_types<32>(a);
        case 64: return recurrent_dispatch_types<64>(a);
        default: return recurrent_dispatch_types<128>(a);
    }
}

}  // namespace efla
