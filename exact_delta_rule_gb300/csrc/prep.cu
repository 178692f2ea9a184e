// Per-token prep: key norm, gate, and the gate-scaled key and value rows.
//
//   lambda_t = ||k_t||^2
//     ["Exact Flow Linear Attention" (gist.science), Metodologia 2]
//   alpha_t  = (1 - e^{-beta_t lambda_t}) / lambda_t  (beta_t at lambda_t = 0;
//              beta_t for the delta-rule update)
//     [same page, Metodologia 3; "Error-Free Linear Attention is a Free Lunch"
//      (howistudyai), Step 1]
//   ak_t = alpha_t k_t,  av_t = alpha_t v_t   (the two factors of the rank-1 write
//     alpha k v^T and of the erase alpha k k^T, in the input dtype)
//
// Each warp handles four token-head rows and issues all their loads before any
// arithmetic; each lane owns d/32 consecutive elements, so a row is one
// contiguous warp access.  Pure streaming: every input byte is read once and
// every output byte written once.
#include "internal.cuh"

namespace efla {
namespace {

template <typename T, int N>
struct alignas(sizeof(T) * N) Vec {
    T x[N];
};

constexpr int RPW = 4;  // rows per warp: all of a warp's loads are in flight before any arithmetic

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(256) prep_kernel(const TIn *__restrict__ k, const TIn *__restrict__ v,
                                                   const float *__restrict__ beta, float *__restrict__ lam_out,
                                                   float *__restrict__ alpha_out, TIn *__restrict__ ak,
                                                   TIn *__restrict__ av, long long n, int euler) {
    constexpr int EK = DK / 32, EV = DV / 32;
    const int lane = threadIdx.x & 31;
    const long long row0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * RPW;
    Vec<TIn, EK> kv[RPW];
    Vec<TIn, EV> vv[RPW];
    float bt[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {  // (row < n is uniform across the warp)
        const long long row = row0 + i;
        if (row < n) {
            kv[i] = reinterpret_cast<const Vec<TIn, EK> *>(k + row * DK)[lane];
            if (av) vv[i] = reinterpret_cast<const Vec<TIn, EV> *>(v + row * DV)[lane];
            bt[i] = beta[row];
        }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const long long row = row0 + i;
        if (row >= n) break;
        float kf[EK];
        float lam = 0.f;
#pragma unroll
        for (int e = 0; e < EK; ++e) {
            kf[e] = to_f32(kv[i].x[e]);
            lam = fmaf(kf[e], kf[e], lam);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
        const float a = efla_alpha(bt[i], lam, euler);
        if (lane == 0) {
            if (lam_out) lam_out[row] = lam;
            if (alpha_out) alpha_out[row] = a;
        }
        if (ak) {
            Vec<TIn, EK> o;
#pragma unroll
            for (int e = 0; e < EK; ++e) o.x[e] = from_f32<TIn>(a * kf[e]);
            reinterpret_cast<Vec<TIn, EK> *>(ak + row * DK)[lane] = o;
        }
        if (av) {
            Vec<TIn, EV> o;
#pragma unroll
            for (int e = 0; e < EV; ++e) o.x[e] = from_f32<TIn>(a * to_f32(vv[i].x[e]));
            reinterpret_cast<Vec<TIn, EV> *>(av + row * DV)[lane] = o;
        }
    }
}

template <int DK, int DV, typename TIn>
cudaError_t prep_launch(const PrepArgs &a) {
    const long long blocks = (a.n + 8 * RPW - 1) / (8 * RPW);
    prep_kernel<DK, DV, TIn><<<(unsigned)blocks, 256, 0, a.stream>>>(
        static_cast<const TIn *>(a.k), static_cast<const TIn *>(a.v), a.beta, a.lam, a.alpha,
        static_cast<TIn *>(a.ak), static_cast<TIn *>(a.av), a.n, a.euler);
    return cudaGetLastError();
}

template <int DK, typename TIn>
cudaError_t prep_dv(const PrepArgs &a) {
    switch (a.dv) {
        case 32: return prep_launch<DK, 32, TIn>(a);
        case 64: return prep_launch<DK, 64, TIn>(a);
        default: return prep_launch<DK, 128, TIn>(a);
    }
}

template <typename TIn>
cudaError_t prep_dk(const PrepArgs &a) {
    switch (a.dk) {
        case 32: return prep_dv<32, TIn>(a);
        case 64: return prep_dv<64, TIn>(a);
        default: return prep_dv<128, TIn>(a);
    }
}

}  // namespace

cudaError_t launch_prep(const PrepArgs &a) {
    if (a.n == 0) return cudaSuccess;
    return a.dtype == EFLA_BF16 ? prep_dk<__nv_bfloat16>(a) : prep_dk<float>(a);
}

}  // namespace efla
