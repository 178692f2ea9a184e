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
// One CTA of 1024 threads per (sequence, head), fp32 on CUDA cores.  S and G live
// in shared memory (rows padded to DV + 1 floats).  A forward sweep leaves u_t of
// every token in the dv output (the reverse sweep overwrites it with dv_t after
// reading it) and S_T in shared memory; the reverse sweep rebuilds
// S_{t-1} = S_t - k_t u_t^T token by token.  Row sums (over d_v) use the mapping
// thread = (row, column group), column sums (over d_k) thread = (column, row
// group); both walk shared memory without bank conflicts.
#include "internal.cuh"

namespace efla {
namespace {

constexpr int NT = 1024;

// d alpha / d beta and d alpha / d lambda (fp32; series in z = beta*lambda where the
// difference form cancels).
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

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(NT) bwd_kernel(const BwdArgs a) {
    constexpr int LD = DV + 1;
    constexpr int CGR = NT / DK, CPR = DV / CGR;  // row mapping: column groups per row, columns each
    constexpr int RGC = NT / DV, RPC = DK / RGC;  // column mapping: row groups per column, rows each
    extern __shared__ float smf[];
    float *S = smf, *G = S + DK * LD;
    float *qs = G + DK * LD, *ks = qs + DK, *vs = ks + DK, *dos = vs + DV, *us = dos + DV, *dxs = us + DV;
    float *rr = dxs + DV;        // [2][CGR][DK] row partials
    float *rc = rr + 2 * CGR * DK;  // [2][RGC][DV] column partials
    float *sc = rc + 2 * RGC * DV;  // [8] scalars, [NT / 32] warp partials

    const TIn *q = static_cast<const TIn *>(a.q), *k = static_cast<const TIn *>(a.k),
              *v = static_cast<const TIn *>(a.v);
    const int unit = blockIdx.x, b = unit / a.H, h = unit % a.H;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int ri = tid % DK, cg = tid / DK;   // row mapping
    const int cj = tid % DV, rg = tid / DV;   // column mapping
    const size_t mat = (size_t)DK * DV;
    const int T = a.T;
    auto rowidx = [&](int t) { return ((size_t)b * T + t) * a.H + h; };

    // S = S0
    for (int e = tid; e < DK * DV; e += NT) {
        const int i = e / DV, j = e % DV;
        S[i * LD + j] = a.S0 ? a.S0[(size_t)unit * mat + e] : 0.f;
    }
    __syncthreads();
    // ------------------------------------------------------------ forward sweep
    // (each token's inputs are loaded one token ahead, so their latency is hidden)
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
        if (tid < DK) ks[tid] = kn;
        if (tid < DV) vs[tid] = vn;
        const float bcur = bn;
        __syncthreads();
        if (t + 1 < T) fetch_f(t + 1);
        if (wid == 0) {
            float lam = 0.f;
            for (int i = lane; i < DK; i += 32) lam = fmaf(ks[i], ks[i], lam);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
            if (lane == 0) sc[0] = efla_alpha(bcur, lam, a.euler);
        }
        float xp = 0.f;  // x_j over this thread's rows
#pragma unroll 8
        for (int i = rg * RPC; i < (rg + 1) * RPC; ++i) xp = fmaf(S[i * LD + cj], ks[i], xp);
        rc[rg * DV + cj] = xp;
        __syncthreads();
        if (tid < DV) {
            float x = 0.f;
#pragma unroll
            for (int g = 0; g < RGC; ++g) x += rc[g * DV + tid];
            const float u = sc[0] * (vs[tid] - x);
            us[tid] = u;
            a.dv[r * DV + tid] = u;  // kept for the reverse sweep
        }
        __syncthreads();
        for (int i = rg * RPC; i < (rg + 1) * RPC; ++i) S[i * LD + cj] = fmaf(ks[i], us[cj], S[i * LD + cj]);
        __syncthreads();
    }
    // G = dS_T
    for (int e = tid; e < DK * DV; e += NT) {
        const int i = e / DV, j = e % DV;
        G[i * LD + j] = a.dST ? a.dST[(size_t)unit * mat + e] : 0.f;
    }
    __syncthreads();
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
            un = a.dv[r * DV + tid];  // u_t, left by this same thread in the forward sweep
        }
        if (tid == 0) bn = a.beta[r];
    };
    if (T > 0) fetch_r(T - 1);
    for (int t = T - 1; t >= 0; --t) {
        const size_t r = rowidx(t);
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
        __syncthreads();
        if (t > 0) fetch_r(t - 1);
        if (wid == 0) {
            float lam = 0.f;
            for (int i = lane; i < DK; i += 32) lam = fmaf(ks[i], ks[i], lam);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
            if (lane == 0) {
                const float bt = bcur;
                float dfdb, dfdl;
                gate_grad(bt, lam, a.euler, dfdb, dfdl);
                sc[0] = efla_alpha(bt, lam, a.euler);
                sc[1] = dfdb;
                sc[2] = dfdl;
            }
        }
        {  // rows: dq = S_t do; G += q do^T; dk1 = G u; S_{t-1} = S_t - k u^T
            const float qi = qs[ri], ki = ks[ri];
            float dq = 0.f, dk1 = 0.f;
#pragma unroll 8
            for (int j = cg * CPR; j < (cg + 1) * CPR; ++j) {
                const float s = S[ri * LD + j], dj = dos[j], uj = us[j];
                const float g = fmaf(qi, dj, G[ri * LD + j]);
                dq = fmaf(s, dj, dq);
                dk1 = fmaf(g, uj, dk1);
                S[ri * LD + j] = fmaf(-ki, uj, s);
                G[ri * LD + j] = g;
            }
            rr[cg * DK + ri] = dq;
            rr[CGR * DK + cg * DK + ri] = dk1;
        }
        __syncthreads();
        {  // columns: du = G^T k; x = S_{t-1}^T k
            float du = 0.f, x = 0.f;
#pragma unroll 8
            for (int i = rg * RPC; i < (rg + 1) * RPC; ++i) {
                du = fmaf(G[i * LD + cj], ks[i], du);
                x = fmaf(S[i * LD + cj], ks[i], x);
            }
            rc[rg * DV + cj] = du;
            rc[RGC * DV + rg * DV + cj] = x;
        }
        __syncthreads();
        float dap = 0.f;
        if (tid < DV) {
            float du = 0.f, x = 0.f;
#pragma unroll
            for (int g = 0; g < RGC; ++g) {
                du += rc[g * DV + tid];
                x += rc[RGC * DV + g * DV + tid];
            }
            const float al = sc[0];
            a.dv[r * DV + tid] = al * du;
            dxs[tid] = -al * du;
            dap = du * (vs[tid] - x);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dap += __shfl_xor_sync(0xffffffffu, dap, off);
        if (lane == 0) sc[8 + wid] = dap;
        __syncthreads();
        {  // rows: dk2 = S_{t-1} dx; G += k dx^T
            const float ki = ks[ri];
            float dk2 = 0.f;
#pragma unroll 8
            for (int j = cg * CPR; j < (cg + 1) * CPR; ++j) {
                const float dx = dxs[j];
                dk2 = fmaf(S[ri * LD + j], dx, dk2);
                G[ri * LD + j] = fmaf(ki, dx, G[ri * LD + j]);
            }
            rr[CGR * DK + cg * DK + ri] += dk2;
        }
        __syncthreads();
        float da = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) da += sc[8 + w];
        if (tid < DK) {
            float dq = 0.f, dk = 0.f;
#pragma unroll
            for (int g = 0; g < CGR; ++g) {
                dq += rr[g * DK + tid];
                dk += rr[CGR * DK + g * DK + tid];
            }
            a.dq[r * DK + tid] = dq;
            a.dk[r * DK + tid] = fmaf(2.f * da * sc[2], ks[tid], dk);
        }
        if (tid == 0) a.dbeta[r] = da * sc[1];
        __syncthreads();
    }
    if (a.dS0)
        for (int e = tid; e < DK * DV; e += NT) {
            const int i = e / DV, j = e % DV;
            a.dS0[(size_t)unit * mat + e] = G[i * LD + j];
        }
}

template <int DK, int DV>
constexpr size_t bwd_smem() {
    return sizeof(float) * (2 * DK * (DV + 1) + 2 * DK + 4 * DV + 2 * (NT / DK) * DK + 2 * (NT / DV) * DV + 8 + NT / 32);
}

template <int DK, int DV, typename TIn>
cudaError_t bwd_launch(const BwdArgs &a) {
    constexpr size_t smem = bwd_smem<DK, DV>();
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
