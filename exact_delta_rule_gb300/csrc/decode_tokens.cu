// Multi-token decode: m new tokens per sequence appended to a resident state,
// S updated in place.  Equal to m successive single-token decode steps, i.e. to
// the recurrence
//   lambda = ||k||^2,  alpha = -expm1(-beta*lambda)/lambda (beta at lambda = 0),
//   S <- (I - alpha k k^T) S + alpha k v^T,  o = S^T q with the updated S
// ["Exact Flow Linear Attention" (gist.science), Metodologia 3;
//  "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-3 and
//  "Putting it all together (pipeline)"] run over the m tokens in order.
//
// Block form.  Writing S_t = S_0 + sum_{i<=t} k_i u_i^T with
// u_t = alpha_t (v_t - S_{t-1}^T k_t), a block of tokens needs S_0 only through
//   X = S_0^T K^T and Y = S_0^T Q^T       (one pass over S for the whole block)
// after which, per column j of S (d_v index),
//   u_t = alpha_t (v_t - X_t - sum_{i<t} (k_t . k_i) u_i)
//   o_t = Y_t + sum_{i<=t} (q_t . k_i) u_i
// is a short forward substitution over the block, and the state update is the
// rank-block S_0 + K^T U.  S is read from HBM once per call and written once.
//
// One CTA of 256 threads per (b, h); thread (half, j) holds rows
// half*DK/2 .. +DK/2-1 of column j of S in registers.  Blocks of MB = 16 tokens;
// K and Q of a block are staged transposed in shared memory ([d][t], read as
// broadcasts), the Gram terms k_t.k_i and q_t.k_i are formed once per block.
#include "internal.cuh"

namespace efla {
namespace {

constexpr int MB = 16;  // tokens per block

template <int DK, int DV, typename TIn, typename TOut>
__global__ void __launch_bounds__(256, 2) decode_tokens_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                                                            const TIn *__restrict__ v, const float *__restrict__ beta,
                                                            float *__restrict__ S, TOut *__restrict__ o, int m, int H,
                                                            int euler) {
    constexpr int NT = 256;
    constexpr int CPT = DV >= 128 ? 1 : 128 / DV;   // columns per thread-half (1 for DV = 128)
    constexpr int HALVES = 2;
    static_assert(DV * CPT == 128, "thread layout assumes DV * CPT == 128");
    constexpr int RPT = DK / HALVES;                 // rows of S per thread

    __shared__ __align__(16) float kT[DK][MB], qT[DK][MB];
    __shared__ float vs[MB][DV];       // v of the block, then u in place (same thread, same (t, j))
    __shared__ float gkk[MB][MB + 1], gqk[MB][MB + 1];
    __shared__ float al[MB], bs[MB];
    __shared__ float red[2][MB][DV];   // partial X and Y of the other row-slices (starts at zero)

    const int unit = blockIdx.x;  // b * H + h
    const int b = unit / H, h = unit % H;
    const int tid = threadIdx.x;
    const int half = tid / 128, l = tid % 128;
    const int j = l % DV, csub = l / DV;           // column, and which of the CPT row-slices (DV < 128)
    // thread (half, l) holds rows [row0, row0 + RPT/CPT) of column j
    constexpr int R = RPT / CPT;
    const int row0 = half * RPT + csub * R;
    float *Su = S + (size_t)unit * DK * DV;
    for (int e = tid; e < 2 * MB * DV; e += NT) (&red[0][0][0])[e] = 0.f;
    float s[R];
#pragma unroll
    for (int r = 0; r < R; ++r) s[r] = Su[(size_t)(row0 + r) * DV + j];

    for (int t0 = 0; t0 < m; t0 += MB) {
        const int mb = min(MB, m - t0);
        __syncthreads();  // the previous block is finished with the shared arrays
        // stage K^T, Q^T [d][t] (zero past mb), V [t][j], beta: every load in flight before any store
        constexpr int NKQ = MB * DK / NT, NV = MB * DV / NT;
        float kr[NKQ], qr[NKQ], vr[NV];
#pragma unroll
        for (int x = 0; x < NKQ; ++x) {
            const int e = tid + x * NT, t = e / DK, d = e % DK;
            const size_t row = ((size_t)b * m + t0 + t) * H + h;
            kr[x] = t < mb ? to_f32(k[row * DK + d]) : 0.f;
            qr[x] = t < mb ? to_f32(q[row * DK + d]) : 0.f;
        }
#pragma unroll
        for (int x = 0; x < NV; ++x) {
            const int e = tid + x * NT, t = e / DV, c = e % DV;
            vr[x] = t < mb ? to_f32(v[(((size_t)b * m + t0 + t) * H + h) * DV + c]) : 0.f;
        }
        const float br = tid < mb ? beta[((size_t)b * m + t0 + tid) * H + h] : 0.f;
#pragma unroll
        for (int x = 0; x < NKQ; ++x) {
            const int e = tid + x * NT, t = e / DK, d = e % DK;
            kT[d][t] = kr[x];
            qT[d][t] = qr[x];
        }
#pragma unroll
        for (int x = 0; x < NV; ++x) {
            const int e = tid + x * NT;
            vs[e / DV][e % DV] = vr[x];
        }
        if (tid < MB) bs[tid] = br;
        __syncthreads();
        // Gram terms: thread (t, i) for t, i < MB
        {
            const int t = tid / MB, i = tid % MB;
            float a = 0.f, c = 0.f;
#pragma unroll 8
            for (int d = 0; d < DK; ++d) {
                const float ki = kT[d][i];
                a = fmaf(kT[d][t], ki, a);
                c = fmaf(qT[d][t], ki, c);
            }
            gkk[t][i] = a;
            gqk[t][i] = c;
            if (t == i) al[t] = t < mb ? efla_alpha(bs[t], a, euler) : 0.f;
        }
        // X = S_0^T K^T, Y = S_0^T Q^T over this thread's rows
        float xp[MB], yp[MB];
#pragma unroll
        for (int t = 0; t < MB; ++t) xp[t] = yp[t] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float sv = s[r];
            const float4 *kr = reinterpret_cast<const float4 *>(kT[row0 + r]);
            const float4 *qr = reinterpret_cast<const float4 *>(qT[row0 + r]);
#pragma unroll
            for (int t4 = 0; t4 < MB / 4; ++t4) {
                const float4 a = kr[t4], c = qr[t4];
                xp[4 * t4] = fmaf(sv, a.x, xp[4 * t4]);
                xp[4 * t4 + 1] = fmaf(sv, a.y, xp[4 * t4 + 1]);
                xp[4 * t4 + 2] = fmaf(sv, a.z, xp[4 * t4 + 2]);
                xp[4 * t4 + 3] = fmaf(sv, a.w, xp[4 * t4 + 3]);
                yp[4 * t4] = fmaf(sv, c.x, yp[4 * t4]);
                yp[4 * t4 + 1] = fmaf(sv, c.y, yp[4 * t4 + 1]);
                yp[4 * t4 + 2] = fmaf(sv, c.z, yp[4 * t4 + 2]);
                yp[4 * t4 + 3] = fmaf(sv, c.w, yp[4 * t4 + 3]);
            }
        }
        // partial sums of all but the first row-slice go through shared memory
        if (half == 1 || csub > 0) {
#pragma unroll
            for (int t = 0; t < MB; ++t) {
                atomicAdd(&red[0][t][j], xp[t]);
                atomicAdd(&red[1][t][j], yp[t]);
            }
        }
        __syncthreads();
        if (half == 0 && csub == 0) {  // one thread per column: the forward substitution
            float u[MB];
#pragma unroll
            for (int t = 0; t < MB; ++t) {
                const float x = xp[t] + red[0][t][j], y = yp[t] + red[1][t][j];
                red[0][t][j] = 0.f;  // cleared for the next block
                red[1][t][j] = 0.f;
                float acc = vs[t][j] - x;
#pragma unroll
                for (int i = 0; i < t; ++i) acc = fmaf(-gkk[t][i], u[i], acc);
                u[t] = al[t] * acc;
                float ov = y;
#pragma unroll
                for (int i = 0; i <= t; ++i) ov = fmaf(gqk[t][i], u[i], ov);
                vs[t][j] = u[t];
                if (t < mb) o[(((size_t)b * m + t0 + t) * H + h) * DV + j] = from_f32<TOut>(ov);
            }
        }
        __syncthreads();
        // S_0 + K^T U over this thread's rows (u of tokens past mb is zero)
        float uc[MB];
#pragma unroll
        for (int t = 0; t < MB; ++t) uc[t] = vs[t][j];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float4 *kr = reinterpret_cast<const float4 *>(kT[row0 + r]);
            float acc = s[r];
#pragma unroll
            for (int t4 = 0; t4 < MB / 4; ++t4) {
                const float4 a = kr[t4];
                acc = fmaf(a.x, uc[4 * t4], acc);
                acc = fmaf(a.y, uc[4 * t4 + 1], acc);
                acc = fmaf(a.z, uc[4 * t4 + 2], acc);
                acc = fmaf(a.w, uc[4 * t4 + 3], acc);
            }
            s[r] = acc;
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) Su[(size_t)(row0 + r) * DV + j] = s[r];
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
