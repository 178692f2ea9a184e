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
// One CTA of 256 threads per (b, h).  Thread (rg, cl) holds rows rg*RW .. +RW-1 and the
// two adjacent columns 2cl, 2cl+1 of S in registers, so each broadcast load of a K^T or Q^T
// row feeds two columns.  Blocks of MB = 16 tokens; K and Q of a block are staged transposed
// in shared memory ([d][t], read as broadcasts), the Gram terms k_t.k_i and q_t.k_i are
// formed once per block, and the partial sums of X and Y of every row group are added in a
// shared-memory pass (no atomics).
#include "internal.cuh"

namespace efla {
namespace {

constexpr int MB = 16;  // tokens per block
constexpr int KS = MB + 4;  // row stride of the staged K^T, Q^T: rows stay 16-byte aligned and the
                            // transposing stores (consecutive d, one t) spread over 8 banks
constexpr int NT = 256;
constexpr int CW = 2;   // columns of S per thread
constexpr size_t PART_BYTES = 2 * (size_t)NT * CW * MB * sizeof(float);  // [2][NRG][MB][DV] (64 KB)

template <int DK, int DV, typename TIn, typename TOut>
__global__ void __launch_bounds__(256, 2) decode_tokens_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                                                            const TIn *__restrict__ v, const float *__restrict__ beta,
                                                            float *__restrict__ S, TOut *__restrict__ o, int m, int H,
                                                            int euler) {
    constexpr int NCL = DV / CW;   // column lanes per row group
    constexpr int NRG = NT / NCL;  // row groups
    constexpr int RW = DK / NRG;   // rows of S per thread
    static_assert(NCL * NRG == NT && RW * NRG == DK && RW >= 1, "thread layout");
    static_assert(2 * NRG * MB * DV * sizeof(float) == PART_BYTES, "partial-sum buffer size");

    __shared__ __align__(16) float kT[DK][KS], qT[DK][KS];
    __shared__ __align__(16) float vs[MB][DV];  // v of the block, then u in place (same thread, same (t, j))
    __shared__ float gkk[MB][MB + 1], gqk[MB][MB + 1];
    __shared__ float al[MB], bs[MB];
    extern __shared__ __align__(16) float part[];  // [X, Y][row group][t][j]; group 0 then holds the sums

    const int unit = blockIdx.x;  // b * H + h
    const int b = unit / H, h = unit % H;
    const int tid = threadIdx.x;
    const int cl = tid % NCL, rg = tid / NCL;
    const int c0 = cl * CW, r0 = rg * RW;
    float *Su = S + (size_t)unit * DK * DV;
    float s[RW][CW];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const float2 x = *reinterpret_cast<const float2 *>(Su + (size_t)(r0 + r) * DV + c0);
        s[r][0] = x.x;
        s[r][1] = x.y;
    }

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
        // Gram terms k_t.k_i, q_t.k_i: thread (t, i4, dq) forms i = 4 i4 .. 4 i4 + 3 over the
        // quarter dq of d (rotated by 2 dq rows so that the four quarters hit different banks),
        // and the four quarters are added across lanes
        {
            static_assert(MB == 16 && NT == 256, "Gram thread layout");
            const int t = tid >> 4, i4 = (tid >> 2) & 3, dq = tid & 3;
            constexpr int DQ = DK / 4;
            float a[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int dd = 0; dd < DQ; ++dd) {
                const int d = dq * DQ + ((dd + 2 * dq) & (DQ - 1));
                const float kt = kT[d][t], qt = qT[d][t];
                const float4 ki = *reinterpret_cast<const float4 *>(&kT[d][4 * i4]);
                const float kv[4] = {ki.x, ki.y, ki.z, ki.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a[e] = fmaf(kt, kv[e], a[e]);
                    c[e] = fmaf(qt, kv[e], c[e]);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                a[e] += __shfl_xor_sync(0xffffffffu, a[e], 1);
                a[e] += __shfl_xor_sync(0xffffffffu, a[e], 2);
                c[e] += __shfl_xor_sync(0xffffffffu, c[e], 1);
                c[e] += __shfl_xor_sync(0xffffffffu, c[e], 2);
            }
            if (dq == 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    gkk[t][4 * i4 + e] = a[e];
                    gqk[t][4 * i4 + e] = c[e];
                }
                if ((t >> 2) == i4) {
                    const int e = t & 3;
                    const float lam = e == 0 ? a[0] : e == 1 ? a[1] : e == 2 ? a[2] : a[3];
                    al[t] = t < mb ? efla_alpha(bs[t], lam, euler) : 0.f;
                }
            }
        }
        // X = S_0^T K^T, then Y = S_0^T Q^T, over this thread's rows: partial sums per row group
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const float(*src)[KS] = pass == 0 ? kT : qT;
            float acc[MB][CW];
#pragma unroll
            for (int t = 0; t < MB; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float4 *row = reinterpret_cast<const float4 *>(src[r0 + r]);
#pragma unroll
                for (int t4 = 0; t4 < MB / 4; ++t4) {
                    const float4 a = row[t4];
                    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[4 * t4 + e][0] = fmaf(s[r][0], av[e], acc[4 * t4 + e][0]);
                        acc[4 * t4 + e][1] = fmaf(s[r][1], av[e], acc[4 * t4 + e][1]);
                    }
                }
            }
            float *dst = part + ((size_t)(pass * NRG + rg) * MB) * DV + c0;
#pragma unroll
            for (int t = 0; t < MB; ++t)
                *reinterpret_cast<float2 *>(dst + t * DV) = make_float2(acc[t][0], acc[t][1]);
        }
        __syncthreads();
        // sums over the row groups into group 0 (each entry owned by one thread)
        for (int e = tid; e < 2 * MB * DV; e += NT) {
            const int pass = e / (MB * DV), rest = e % (MB * DV);
            float *p0 = part + (size_t)pass * NRG * MB * DV + rest;
            float acc = p0[0];
#pragma unroll
            for (int g = 1; g < NRG; ++g) acc += p0[(size_t)g * MB * DV];
            p0[0] = acc;
        }
        __syncthreads();
        if (tid < DV) {  // one thread per column: the forward substitution
            const int j = tid;
            const float *X = part, *Y = part + (size_t)NRG * MB * DV;
            float u[MB];
#pragma unroll
            for (int t = 0; t < MB; ++t) {
                float acc = vs[t][j] - X[t * DV + j];
#pragma unroll
                for (int i = 0; i < t; ++i) acc = fmaf(-gkk[t][i], u[i], acc);
                u[t] = al[t] * acc;
                float ov = Y[t * DV + j];
#pragma unroll
                for (int i = 0; i <= t; ++i) ov = fmaf(gqk[t][i], u[i], ov);
                vs[t][j] = u[t];
                if (t < mb) o[(((size_t)b * m + t0 + t) * H + h) * DV + j] = from_f32<TOut>(ov);
            }
        }
        __syncthreads();
        // S_0 + K^T U over this thread's rows (u of tokens past mb is zero)
        float uc[MB][CW];
#pragma unroll
        for (int t = 0; t < MB; ++t) {
            const float2 x = *reinterpret_cast<const float2 *>(&vs[t][c0]);
            uc[t][0] = x.x;
            uc[t][1] = x.y;
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const float4 *row = reinterpret_cast<const float4 *>(kT[r0 + r]);
            float a0 = s[r][0], a1 = s[r][1];
#pragma unroll
            for (int t4 = 0; t4 < MB / 4; ++t4) {
                const float4 a = row[t4];
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a0 = fmaf(av[e], uc[4 * t4 + e][0], a0);
                    a1 = fmaf(av[e], uc[4 * t4 + e][1], a1);
                }
            }
            s[r][0] = a0;
            s[r][1] = a1;
        }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r)
        *reinterpret_cast<float2 *>(Su + (size_t)(r0 + r) * DV + c0) = make_float2(s[r][0], s[r][1]);
}

template <int DK, int DV, typename TIn, typename TOut>
cudaError_t tokens_launch(const DecodeArgs &a) {
    static bool attr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr[dev]) {
        e = cudaFuncSetAttribute(decode_tokens_kernel<DK, DV, TIn, TOut>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)PART_BYTES);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr[dev] = true;
    }
    decode_tokens_kernel<DK, DV, TIn, TOut><<<a.B * a.H, NT, PART_BYTES, a.stream>>>(
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
