// Eager (load-update-store) baselines: the conventional decode step that
// reads and writes the whole state at each step (the thread's post [2/N] of
// "Songlin Yang releases ReplaySSM, cutting hybrid SSM memory traffic in half
// ..."; the abstract's "eager state management"), and the per-draft snapshot
// scheme for speculative decoding (post [3/N] of the same thread: one state
// kept per draft token so that any accepted prefix can be resumed).
//
// Same slab geometry and streaming as the replay kernels, so the comparison
// isolates the algorithm: one CTA per HPC heads of one sequence, the fp32
// slab held in registers, updated in place and stored after every draft.
//   Mamba-2: S <- alpha S + (dt x) k^T, y = S q + D x  (row-local update)
//   GDN:     a = S k, u = beta (v - alpha a), S <- alpha S + u k^T,
//            y = S_new q = alpha (S q) + u (k . q)
//   KDA (one decay per key channel): a = S (alpha (.) k), u = beta (v - a),
//            S <- S diag(alpha) + u k^T, y = S (alpha (.) q) + u (k . q)
#include "rs_common.cuh"
#include "rs_internal.h"

namespace rs {

template <int KIND, int P, int N, int HPC, int NT>
__global__ void __launch_bounds__(NT) eager_kernel(const EagerParams p) {
    using Gm = Geo<P, N, NT, float>;
    constexpr int VEC = Gm::VEC, TPR = Gm::TPR, R = Gm::R;
    constexpr bool KDA = KIND == RS_KDA;
    constexpr int J1 = KIND != RS_MAMBA2 ? 2 : 1;
    extern __shared__ __align__(16) float sm[];
    float *kq = sm;                              // [2*kMaxT][N]: k_i rows 0.., q_i rows kMaxT..
    float *vv = kq + 2 * kMaxT * N;              // [HPC][kMaxT][P]: Mamba-2 dt*x, GDN v
    float *sc = vv + HPC * kMaxT * P;            // [HPC][kMaxT][2]: alpha, beta
    float *kqd = sc + HPC * kMaxT * 2;           // [kMaxT] k_i . q_i (GDN)
    float *uu = kqd + kMaxT;                     // [HPC][P] GDN u of the current draft
    float *red = uu + HPC * P;                   // [NW][HPC*J1][P]
    float *av = red + (NT / 32) * HPC * J1 * P;  // KDA: [HPC][kMaxT][N] decay vectors

    const int tid = threadIdx.x;
    const int b = blockIdx.y, h0 = blockIdx.x * HPC;
    const int H = p.H, G = p.G, T = p.T;
    const int g = h0 / (H / G);
    const int pv = tid % TPR, n0 = (tid / TPR) * R, p0 = pv * VEC;
    const size_t slab = (size_t)N * P;
    const int cur = p.cur ? p.cur[b] : 0;
    if (cur < 0 || cur >= p.slots) return;  // not a pool slot: leave the sequence alone

    uint4 tile[HPC][R];
#pragma unroll
    for (int hd = 0; hd < HPC; ++hd) {
        const float *src = p.S + (((size_t)b * p.slots + cur) * H + h0 + hd) * slab + (size_t)n0 * P + p0;
#pragma unroll
        for (int k = 0; k < R; ++k) tile[hd][k] = ld_stream(src + (size_t)k * P);
    }

    // stage the drafts' keys / queries and per-head scalars
    for (int rr = tid / 8; rr < 2 * T; rr += NT / 8) {
        const int i = rr % T;
        const bool isq = rr >= T;
        const uint16_t *src = (KIND == RS_MAMBA2 ? (isq ? p.Cm : p.Bm) : (isq ? p.q : p.k)) +
                              (((size_t)b * T + i) * G + g) * N;
        bf16_row_to_smem(kq + (size_t)(isq ? kMaxT + i : i) * N, src, N, tid % 8, 8);
    }
    for (int it = tid; it < HPC * T * P; it += NT) {
        const int pp = it % P, i = (it / P) % T, hd = it / (P * T), hh = h0 + hd;
        const size_t bti = ((size_t)b * T + i) * H + hh;
        const uint16_t *src = KIND == RS_MAMBA2 ? p.x : p.v;
        const float xv = bf2f(src[bti * P + pp]);
        vv[(hd * kMaxT + i) * P + pp] = KIND == RS_MAMBA2 ? p.dt[bti] * xv : xv;
    }
    if (KDA) {
        for (int it = tid; it < HPC * T * N; it += NT) {
            const int n = it % N, i = (it / N) % T, hd = it / (N * T), hh = h0 + hd;
            av[((size_t)hd * kMaxT + i) * N + n] = p.alpha[(((size_t)b * T + i) * H + hh) * N + n];
        }
    }
    for (int it = tid; it < HPC * T; it += NT) {
        const int i = it % T, hd = it / T, hh = h0 + hd;
        const size_t bti = ((size_t)b * T + i) * H + hh;
        if (KIND == RS_MAMBA2) {
            sc[(hd * kMaxT + i) * 2] = expf(p.dt[bti] * p.A[hh]);
        } else {
            sc[(hd * kMaxT + i) * 2] = KDA ? 1.f : p.alpha[bti];
            sc[(hd * kMaxT + i) * 2 + 1] = p.beta[bti];
        }
    }
    __syncthreads();
    if (KIND != RS_MAMBA2) {  // k_i . q_i, one warp per draft
        const int w = tid / 32, lane = tid % 32;
        for (int i = w; i < T; i += NT / 32) {
            float a = 0.f;
            for (int n = lane; n < N; n += 32) a += kq[(size_t)i * N + n] * kq[(size_t)(kMaxT + i) * N + n];
#pragma unroll
            for (int off = 16; off; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            if (lane == 0) kqd[i] = a;
        }
        __syncthreads();
    }

    for (int i = 0; i < T; ++i) {
        const float *kvec = kq + (size_t)i * N + n0;
        const float *qvec = kq + (size_t)(kMaxT + i) * N + n0;
        float acc[HPC * J1][VEC];
#pragma unroll
        for (int a = 0; a < HPC * J1; ++a)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[a][e] = 0.f;

        if (KIND == RS_MAMBA2) {
#pragma unroll
            for (int hd = 0; hd < HPC; ++hd) {
                const float al = sc[(hd * kMaxT + i) * 2];
                const float4 v4 = *reinterpret_cast<const float4 *>(vv + (hd * kMaxT + i) * P + p0);
                const float vloc[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    float s[VEC];
                    unpack<float, VEC>(tile[hd][k], s);
                    const float kn = kvec[k], qn = qvec[k];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        s[e] = fmaf(al, s[e], vloc[e] * kn);
                        acc[hd][e] = fmaf(s[e], qn, acc[hd][e]);
                    }
                    tile[hd][k] = make_uint4(__float_as_uint(s[0]), __float_as_uint(s[1]),
                                             __float_as_uint(s[2]), __float_as_uint(s[3]));
                }
            }
            cta_reduce<NT, TPR, VEC, P, HPC * J1>(acc, HPC * J1, red);
            for (int it = tid; it < HPC * P; it += NT) {
                const int pp = it % P, hd = it / P, hh = h0 + hd;
                const size_t bti = ((size_t)b * T + i) * H + hh;
                const float Dh = p.D ? p.D[hh] : 0.f;
                p.y[bti * P + pp] = red[(size_t)hd * P + pp] + Dh * bf2f(p.x[bti * P + pp]);
            }
        } else {
#pragma unroll
            for (int hd = 0; hd < HPC; ++hd)
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    float s[VEC];
                    unpack<float, VEC>(tile[hd][k], s);
                    // KDA: S diag(alpha) k and S diag(alpha) q
                    const float an = KDA ? av[((size_t)hd * kMaxT + i) * N + n0 + k] : 1.f;
                    const float kn = kvec[k] * an, qn = qvec[k] * an;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        acc[hd * 2][e] = fmaf(s[e], kn, acc[hd * 2][e]);
                        acc[hd * 2 + 1][e] = fmaf(s[e], qn, acc[hd * 2 + 1][e]);
                    }
                }
            cta_reduce<NT, TPR, VEC, P, HPC * J1>(acc, HPC * J1, red);
            for (int it = tid; it < HPC * P; it += NT) {
                const int pp = it % P, hd = it / P, hh = h0 + hd;
                const size_t bti = ((size_t)b * T + i) * H + hh;
                const float al = sc[(hd * kMaxT + i) * 2], be = sc[(hd * kMaxT + i) * 2 + 1];
                const float a = red[(size_t)(hd * 2) * P + pp], bq = red[(size_t)(hd * 2 + 1) * P + pp];
                const float u = be * (vv[(hd * kMaxT + i) * P + pp] - al * a);
                uu[hd * P + pp] = u;
                p.y[bti * P + pp] = fmaf(al, bq, u * kqd[i]);
            }
            __syncthreads();
#pragma unroll
            for (int hd = 0; hd < HPC; ++hd) {
                const float al = sc[(hd * kMaxT + i) * 2];
                const float4 u4 = *reinterpret_cast<const float4 *>(uu + hd * P + p0);
                const float uloc[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    float s[VEC];
                    unpack<float, VEC>(tile[hd][k], s);
                    const float kn = kvec[k];
                    const float ar = KDA ? av[((size_t)hd * kMaxT + i) * N + n0 + k] : al;  // this row's decay
#pragma unroll
                    for (int e = 0; e < VEC; ++e) s[e] = fmaf(ar, s[e], uloc[e] * kn);
                    tile[hd][k] = make_uint4(__float_as_uint(s[0]), __float_as_uint(s[1]),
                                             __float_as_uint(s[2]), __float_as_uint(s[3]));
                }
            }
        }
        // store this draft's state (in place for a plain step)
        const int dst_slot = (cur + 1 + i) % p.slots;
#pragma unroll
        for (int hd = 0; hd < HPC; ++hd) {
            float *dst = p.S + (((size_t)b * p.slots + dst_slot) * H + h0 + hd) * slab + (size_t)n0 * P + p0;
#pragma unroll
            for (int k = 0; k < R; ++k) st_stream(dst + (size_t)k * P, tile[hd][k]);
        }
        __syncthreads();  // the next draft's reduction reuses red / uu
    }
}

template <int KIND, int P, int N, int HPC, int NT>
static cudaError_t launch_eager(const EagerParams &p, cudaStream_t s) {
    constexpr int J1 = KIND != RS_MAMBA2 ? 2 : 1;
    const size_t floats = 2 * kMaxT * N + HPC * kMaxT * P + HPC * kMaxT * 2 + kMaxT + HPC * P +
                          (NT / 32) * HPC * J1 * P + (KIND == RS_KDA ? HPC * kMaxT * N : 0);
    const size_t smem = floats * sizeof(float);
    auto kern = eager_kernel<KIND, P, N, HPC, NT>;
    static SmemGrants grants;  // this instantiation's opt-in, per device
    const cudaError_t e = grant_smem(reinterpret_cast<const void *>(kern), (int)smem, grants);
    if (e != cudaSuccess) return e;
    kern<<<dim3(p.H / HPC, p.B), NT, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t eager_launch(const EagerParams &p, int kind, int P, int N, cudaStream_t s) {
    const bool two = (p.H / p.G) % 2 == 0;
    if (kind == RS_MAMBA2) {
        if (P == 64 && N == 128) return two ? launch_eager<RS_MAMBA2, 64, 128, 2, 256>(p, s)
                                            : launch_eager<RS_MAMBA2, 64, 128, 1, 256>(p, s);
        if (P == 64 && N == 64) return two ? launch_eager<RS_MAMBA2, 64, 64, 2, 128>(p, s)
                                           : launch_eager<RS_MAMBA2, 64, 64, 1, 128>(p, s);
    } else if (kind == RS_GDN) {
        if (P == 128 && N == 128) return launch_eager<RS_GDN, 128, 128, 1, 256>(p, s);
        if (P == 64 && N == 64) return launch_eager<RS_GDN, 64, 64, 1, 128>(p, s);
    } else {
        if (P == 128 && N == 128) return launch_eager<RS_KDA, 128, 128, 1, 256>(p, s);
        if (P == 64 && N == 64) return launch_eager<RS_KDA, 64, 64, 1, 128>(p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rs
