// Multi-token decode: m new tokens per sequence appended to a resident state,
// S updated in place.  Equal to m successive single-token decode steps, i.e. to
// the recurrence
//   lambda = ||k||^2,  alpha = -expm1(-beta*lambda)/lambda (beta at lambda = 0),
//   S <- (I - alpha k k^T) S + alpha k v^T,  o = S^T q with the updated S
// ["Exact Flow Linear Attention" (gist.science), Metodologia 3;
//  "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-3 and
//  "Putting it all together (pipeline)"] run over the m tokens in order.
//
// One CTA of 256 threads per (b, h).  S[b,h] is read into registers once, the
// m updates are applied there, and S is written back once, so HBM traffic is
// that of one decode step plus the m tokens' q, k, v, beta and o.  Per token the
// single-pass form x = S^T k, y = S^T q, u = alpha (v - x), o = y + (q.k) u,
// S += k u^T is used (S_new^T q = S^T q + u (k.q)).  The next token's inputs
// are loaded while the current one is processed; k, q, u and the per-token
// scalars are double-buffered in shared memory, so three CTA barriers per token
// suffice.
#include "internal.cuh"

namespace efla {
namespace {

template <int DK, int DV, typename TIn, typename TOut>
__global__ void __launch_bounds__(256) decode_tokens_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                                                            const TIn *__restrict__ v, const float *__restrict__ beta,
                                                            float *__restrict__ S, TOut *__restrict__ o, int m, int H,
                                                            int euler) {
    constexpr int CG = DV / 4;      // column groups of 4 floats (lanes along d_v)
    constexpr int RG = 256 / CG;    // row groups
    constexpr int ROWS = DK / RG;   // rows of S per thread
    static_assert(ROWS >= 1 && DK % RG == 0, "unsupported decode shape");

    __shared__ float ks[2][DK], qs[2][DK], us[2][DV];
    __shared__ float red_x[RG][DV], red_y[RG][DV];
    __shared__ float scal[2][2];

    const int unit = blockIdx.x;  // b * H + h
    const int b = unit / H, h = unit % H;
    const int tid = threadIdx.x;
    const int cg = tid % CG, rg = tid / CG;
    auto row_of = [&](int t) { return ((size_t)b * m + t) * H + h; };

    float4 *Su = reinterpret_cast<float4 *>(S + (size_t)unit * DK * DV);
    float4 reg[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) reg[r] = Su[(size_t)(rg + r * RG) * CG + cg];

    float kn = 0.f, qn = 0.f, vn = 0.f, bn = 0.f;  // the next token's inputs
    auto fetch = [&](int t) {
        const size_t r = row_of(t);
        if (tid < DK) {
            kn = to_f32(k[r * DK + tid]);
            qn = to_f32(q[r * DK + tid]);
        }
        if (tid < DV) vn = to_f32(v[r * DV + tid]);
        if (tid == 0) bn = beta[r];
    };
    fetch(0);

    for (int t = 0; t < m; ++t) {
        const int pb = t & 1;
        if (tid < DK) {
            ks[pb][tid] = kn;
            qs[pb][tid] = qn;
        }
        const float vcur = vn, bcur = bn;
        __syncthreads();  // k, q of token t visible; token t-1's reductions consumed
        if (t + 1 < m) fetch(t + 1);
        if (tid < 32) {
            float lam = 0.f, qk = 0.f;
            for (int i = tid; i < DK; i += 32) {
                lam = fmaf(ks[pb][i], ks[pb][i], lam);
                qk = fmaf(qs[pb][i], ks[pb][i], qk);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                lam += __shfl_xor_sync(0xffffffffu, lam, off);
                qk += __shfl_xor_sync(0xffffffffu, qk, off);
            }
            if (tid == 0) {
                scal[pb][0] = efla_alpha(bcur, lam, euler);
                scal[pb][1] = qk;
            }
        }
        float px[4] = {0.f, 0.f, 0.f, 0.f}, py[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float ki = ks[pb][rg + r * RG], qi = qs[pb][rg + r * RG];
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
        __syncthreads();  // partial sums and the token's scalars visible
        if (tid < DV) {
            float x = 0.f, y = 0.f;
#pragma unroll 8
            for (int r = 0; r < RG; ++r) {
                x += red_x[r][tid];
                y += red_y[r][tid];
            }
            const float u = scal[pb][0] * (vcur - x);
            us[pb][tid] = u;
            o[row_of(t) * DV + tid] = from_f32<TOut>(fmaf(scal[pb][1], u, y));
        }
        __syncthreads();  // u of token t visible
        const float u0 = us[pb][cg * 4 + 0], u1 = us[pb][cg * 4 + 1], u2 = us[pb][cg * 4 + 2],
                    u3 = us[pb][cg * 4 + 3];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float ki = ks[pb][rg + r * RG];
            reg[r].x = fmaf(ki, u0, reg[r].x);
            reg[r].y = fmaf(ki, u1, reg[r].y);
            reg[r].z = fmaf(ki, u2, reg[r].z);
            reg[r].w = fmaf(ki, u3, reg[r].w);
        }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) Su[(size_t)(rg + r * RG) * CG + cg] = reg[r];
}

template <int DK, int DV, typename TIn, typename TOut>
cudaError_t tokens_launch(const DecodeArgs &a) {
    decode_tokens_kernel<DK, DV, TIn, TOut><<<a.B * a.H, 256, 0, a.stream>>>(
        static_cast<const TIn *>(a.q), static_cast<const TIn *>(a.k), static_cast<const TIn *>(a.v), a.beta, a.S,
        static_cast<TOut *>(a.o), a.m, a.H, a.euler);
    return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t tokens_types(const DecodeArgs &a) {
    const bool ib = a.in_dtype == EFLA_BF16, ob = a.o_dtype == EFLA_BF16;
    if (ib && ob) return tokens_launch<DK, DV, __nv_bfloat16, __nv_bfloat16>(a);
    if (ib) return tokens_launch<DK, DV, __nv_bfloat16, float>(a);
    if (ob) return tokens_launch<DK, DV, float, __nv_bfloat16>(a);
    return tokens_launch<DK, DV, float, float>(a);
}

template <int DK>
cudaError_t tokens_dv(const DecodeArgs &a) {
    switch (a.dv) {
        case 32: return tokens_types<DK, 32>(a);
        case 64: return tokens_types<DK, 64>(a);
        default: return tokens_types<DK, 128>(a);
    }
}

}  // namespace

cudaError_t launch_decode_tokens(const DecodeArgs &a) {
    if (a.B == 0 || a.m == 0) return cudaSuccess;
    switch (a.dk) {
        case 32: return tokens_dv<32>(a);
        case 64: return tokens_dv<64>(a);
        default: return tokens_dv<128>(a);
    }
}

}  // namespace efla
