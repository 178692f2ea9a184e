// Backward pass of the EFLA forward: gradients dq, dk, dv, dbeta, dS0 from the
// gradients do of the outputs and dS_T of the final state.
//
// The pages give no backward formulas; this is reverse mode of the recurrence
//   lambda = ||k||^2, alpha = f(beta, lambda) = -expm1(-beta*lambda)/lambda,
//   x = S_{t-1}^T k, u = alpha (v - x), S_t = S_{t-1} + k u^T, o = S_t^T q
// ["Exact Flow Linear Attention" (gist.science), Metodologia 3; "Error-Free
// Linear Attention is a Free Lunch" (howistudyai), Steps 1-3], in reverse token
// order with G = dL/dS_t:
//   dq = S_t do;  G += q do^T;  du = G^T k;  dk = G u;  dv = alpha du;
//   dalpha = du . (v - x);  dx = -alpha du;  dk += S_{t-1} dx;  G += k dx^T;
//   dbeta = dalpha df/dbeta;  dk += 2 dalpha df/dlambda k;
// and dS0 = G at the start of the sequence.
//
// One CTA of 1024 threads per (sequence, head), fp32 on CUDA cores.  S and G are
// held in registers as a 32 x 32 grid of tiles (thread (ti, tj) = (warp, lane)
// owns rows ti*DK/32.., columns tj*DV/32..), so every per-element update is
// register arithmetic.  Row sums (over d_v) and column sums (over d_k) go through
// shared memory once per tile: each thread writes one partial per row (column)
// of its tile, then DK (DV) threads add the 32 partials of a row (column).
// A forward sweep recomputes the states and leaves u_t of every token in the dv
// output (the reverse sweep reads it back before overwriting it with dv_t); the
// reverse sweep rebuilds S_{t-1} = S_t - k_t u_t^T.  Each token's inputs are
// loaded one token ahead.
#include "internal.cuh"

namespace efla {
namespace {

constexpr int NT = 1024;

template <int DK, int DV>
struct BwdSmem {
    static constexpr int RP = 33;                          // row partials [DK][RP] (padded)
    static constexpr size_t vec = 2 * DK + 4 * DV;         // q, k | v, do, u, dx
    static constexpr size_t rowp = 2 * (size_t)DK * RP;    // two quantities
    static constexpr size_t colp = 2 * 32 * (size_t)DV;    // two quantities
    static constexpr size_t sums = 2 * DK + 2 * DV;
    static constexpr size_t bytes = sizeof(float) * (vec + rowp + colp + sums + 8 + NT / 32);
};

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(NT, 1) bwd_kernel(const BwdArgs a) {
    constexpr int RT = DK / 32, CT = DV / 32;  // tile of S / G per thread
    using L = BwdSmem<DK, DV>;
    extern __shared__ __align__(16) float smf[];
    float *qs = smf, *ks = qs + DK, *vs = ks + DK, *dos = vs + DV, *us = dos + DV, *dxs = us + DV;
    float *rowp = dxs + DV;                 // [2][DK][RP]
    float *colp = rowp + L::rowp;           // [2][32][DV]
    float *rsum = colp + L::colp;           // [2][DK]
    float *csum = rsum + 2 * DK;            // [2][DV]
    float *sc = csum + 2 * DV;              // [8] scalars, [NT/32] warp partials

    const TIn *q = static_cast<const TIn *>(a.q), *k = static_cast<const TIn *>(a.k),
              *v = static_cast<const TIn *>(a.v);
    const int unit = blockIdx.x, b = unit / a.H, h = unit % a.H;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int ti = wid, tj = lane, r0 = ti * RT, c0 = tj * CT;
    const size_t mat = (size_t)DK * DV;
    const int T = a.T;
    auto rowidx = [&](int t) { return ((size_t)b * T + t) * a.H + h; };

    float S[RT][CT], G[RT][CT];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int c = 0; c < CT; ++c) S[r][c] = a.S0 ? a.S0[(size_t)unit * mat + (size_t)(r0 + r) * DV + c0 + c] : 0.f;

    // ------------------------------------------------------------ forward sweep
    float kn = 0.f, vn = 0.f, bn = 0.f;
    auto fetch_f = [&](int t) {
        const size_t r = rowidx(t);
        if (tid < DK) kn = to_f32(k[r * DK + tid]);
        if (tid < DV) vn = to_f32(v[r * DV + tid]);
        if (tid == 0) bn = a.beta[r];
    };
    if (T > 0) fetch_f(0);
    for (int t = 0; t < T; ++t) {
        const size_t r = rowidx(t);
        __syncthreads();  // the previous token's update has read k and u
        if (tid < DK) ks[tid] = kn;
        if (tid < DV) vs[tid] = vn;
        const float bcur = bn;
        __syncthreads();  // this token's k, v visible
        if (t + 1 < T) fetch_f(t + 1);
        if (wid == 0) {
            float lam = 0.f;
            for (int i = lane; i < DK; i += 32) lam = fmaf(ks[i], ks[i], lam);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
            if (lane == 0) sc[0] = efla_alpha(bcur, lam, a.euler);
        }
#pragma unroll
        for (int c = 0; c < CT; ++c) {  // x = S^T k: this tile's column partials
            float px = 0.f;
#pragma unroll
            for (int rr = 0; rr < RT; ++rr) px = fmaf(S[rr][c], ks[r0 + rr], px);
            colp[ti * DV + c0 + c] = px;
        }
        __syncthreads();
        if (tid < DV) {
            float x = 0.f;
#pragma unroll 8
            for (int tt = 0; tt < 32; ++tt) x += colp[tt * DV + tid];
            const float u = sc[0] * (vs[tid] - x);
            us[tid] = u;
            a.dv[r * DV + tid] = u;  // kept for the reverse sweep (read back by this thread)
        }
        __syncthreads();  // u visible
#pragma unroll
        for (int rr = 0; rr < RT; ++rr)
#pragma unroll
            for (int c = 0; c < CT; ++c) S[rr][c] = fmaf(ks[r0 + rr], us[c0 + c], S[rr][c]);
    }
    // G = dS_T
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int c = 0; c < CT; ++c) G[r][c] = a.dST ? a.dST[(size_t)unit * mat + (size_t)(r0 + r) * DV + c0 + c] : 0.f;

    // ------------------------------------------------------------ reverse sweep
    float qn = 0.f, dn = 0.f, un = 0.f;
    auto fetch_r = [&](int t) {
        const size_t r = rowidx(t);
        if (tid < DK) {
            qn = to_f32(q[r * DK + tid]);
            kn = to_f32(k[r * DK + tid]);
        }
        if (tid < DV) {
            vn = to_f32(v[r * DV + tid]);
            dn = a.dO[r * DV + tid];
            un = a.dv[r * DV + tid];  // u_t, written by this same thread in the forward sweep
        }
        if (tid == 0) bn = a.beta[r];
    };
    if (T > 0) fetch_r(T - 1);
    for (int t = T - 1; t >= 0; --t) {
        const size_t r = rowidx(t);
        __syncthreads();  // the previous token is done with every shared array
        if (tid < DK) {
            qs[tid] = qn;
            ks[tid] = kn;
        }
        if (tid < DV) {
            vs[tid] = vn;
            dos[tid] = dn;
            us[tid] = un;
        }
        const float bcur = bn;
        __syncthreads();  // this token's vectors visible
        if (t > 0) fetch_r(t - 1);
        if (wid == 0) {
            float lam = 0.f;
            for (int i = lane; i < DK; i += 32) lam = fmaf(ks[i], ks[i], lam);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
            if (lane == 0) {
                float dfdb, dfdl;
                gate_grad(bcur, lam, a.euler, dfdb, dfdl);
                sc[0] = efla_alpha(bcur, lam, a.euler);
                sc[1] = dfdb;
                sc[2] = dfdl;
            }
        }
        // rows: dq = S_t do; G += q do^T; dk1 = G u; S_{t-1} = S_t - k u^T;
        // then columns: du = G^T k; x = S_{t-1}^T k
        {
            float pdq[RT], pdk[RT];
#pragma unroll
            for (int rr = 0; rr < RT; ++rr) {
                const float qi = qs[r0 + rr], ki = ks[r0 + rr];
                float dq = 0.f, dk1 = 0.f;
#pragma unroll
                for (int c = 0; c < CT; ++c) {
                    const float dj = dos[c0 + c], uj = us[c0 + c];
                    const float g = fmaf(qi, dj, G[rr][c]);
                    dq = fmaf(S[rr][c], dj, dq);
                    dk1 = fmaf(g, uj, dk1);
                    S[rr][c] = fmaf(-ki, uj, S[rr][c]);
                    G[rr][c] = g;
                }
                pdq[rr] = dq;
                pdk[rr] = dk1;
            }
#pragma unroll
            for (int rr = 0; rr < RT; ++rr) {
                rowp[(r0 + rr) * L::RP + tj] = pdq[rr];
                rowp[(DK + r0 + rr) * L::RP + tj] = pdk[rr];
            }
#pragma unroll
            for (int c = 0; c < CT; ++c) {
                float du = 0.f, x = 0.f;
#pragma unroll
                for (int rr = 0; rr < RT; ++rr) {
                    du = fmaf(G[rr][c], ks[r0 + rr], du);
                    x = fmaf(S[rr][c], ks[r0 + rr], x);
                }
                colp[ti * DV + c0 + c] = du;
                colp[(32 + ti) * DV + c0 + c] = x;
            }
        }
        __syncthreads();
        if (tid < 2 * DV) {  // column sums: du, x
            const int qn2 = tid / DV, j = tid % DV;
            float s = 0.f;
#pragma unroll 8
            for (int tt = 0; tt < 32; ++tt) s += colp[(qn2 * 32 + tt) * DV + j];
            csum[qn2 * DV + j] = s;
        }
        if (tid < 2 * DK) {  // row sums: dq, dk1
            const float *pp = rowp + tid * L::RP;
            float s = 0.f;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) s += pp[j];
            rsum[tid] = s;
        }
        __syncthreads();
        float dap = 0.f;
        if (tid < DV) {
            const float du = csum[tid], x = csum[DV + tid], al = sc[0];
            a.dv[r * DV + tid] = al * du;
            dxs[tid] = -al * du;
            dap = du * (vs[tid] - x);
        }
        if (tid < DK) a.dq[r * DK + tid] = rsum[tid];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dap += __shfl_xor_sync(0xffffffffu, dap, off);
        if (lane == 0) sc[8 + wid] = dap;
        __syncthreads();  // dx visible
        {  // rows: dk2 = S_{t-1} dx;  G += k dx^T
#pragma unroll
            for (int rr = 0; rr < RT; ++rr) {
                const float ki = ks[r0 + rr];
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < CT; ++c) {
                    const float dx = dxs[c0 + c];
                    acc = fmaf(S[rr][c], dx, acc);
                    G[rr][c] = fmaf(ki, dx, G[rr][c]);
                }
                rowp[(r0 + rr) * L::RP + tj] = acc;
            }
        }
        __syncthreads();
        if (tid < DK) {
            float da = 0.f;
#pragma unroll
            for (int w = 0; w < (DV + 31) / 32; ++w) da += sc[8 + w];  // only warps holding columns contribute
            const float *pp = rowp + tid * L::RP;
            float dk2 = 0.f;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) dk2 += pp[j];
            a.dk[r * DK + tid] = fmaf(2.f * da * sc[2], ks[tid], rsum[DK + tid] + dk2);
            if (tid == 0) a.dbeta[r] = da * sc[1];
        }
    }
    if (a.dS0) {
#pragma unroll
        for (int rr = 0; rr < RT; ++rr)
#pragma unroll
            for (int c = 0; c < CT; ++c) a.dS0[(size_t)unit * mat + (size_t)(r0 + rr) * DV + c0 + c] = G[rr][c];
    }
}

template <int DK, int DV, typename TIn>
cudaError_t bwd_launch(const BwdArgs &a) {
    constexpr size_t smem = BwdSmem<DK, DV>::bytes;
    static bool attr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr[dev]) {
        e = cudaFuncSetAttribute(bwd_kernel<DK, DV, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr[dev] = true;
    }
    bwd_kernel<DK, DV, TIn><<<(unsigned)(a.B * a.H), NT, smem, a.stream>>>(a);
    return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t bwd_types(const BwdArgs &a) {
    return a.in_dtype == EFLA_BF16 ? bwd_launch<DK, DV, __nv_bfloat16>(a) : bwd_launch<DK, DV, float>(a);
}

template <int DK>
cudaError_t bwd_dv(const BwdArgs &a) {
    switch (a.dv_dim) {
        case 32: return bwd_types<DK, 32>(a);
        case 64: return bwd_types<DK, 64>(a);
        default: return bwd_types<DK, 128>(a);
    }
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs &a) {
    if (a.B == 0) return cudaSuccess;
    switch (a.dk_dim) {
        case 32: return bwd_dv<32>(a);
        case 64: return bwd_dv<64>(a);
        default: return bwd_dv<128>(a);
    }
}

}  // namespace efla
