// Output-only replay kernels of the ReplaySSM decode path (Mamba-2 and Gated
// DeltaNet): standard decode with the flush route fused, speculative verify
// with the fold of committed records fused, forced flush, and materialise.
//
// The state of one (sequence, head) is S = gamma * S_c + sum_r w_r v_r k_r^T
// over the records r since the checkpoint S_c ("ReplaySSM: Cache SSM Inputs,
// Not State", section "How it works").  One CTA owns HPC heads of one
// sequence.  It streams those heads' checkpoint slabs once, with 128-bit
// evict-first loads issued up front into registers, and:
//   * dots the slab with the step's query (and, for GDN, key) vectors: the
//     only work proportional to the state size on a non-flush step;
//   * adds the buffer replay, sum_r w_r (k_r . q) v_r, from the small records
//     staged in shared memory;
//   * on a flush, rewrites the slab from the same registers as
//     gamma * S_c + (V diag(w)) K^T (the rank-F update of the "flush route").
// Checkpoint slabs are stored key-major ([N][P], value index contiguous), so
// every state element's dot products accumulate within its own thread and
// only one CTA-level reduction per launch is needed.
#include "rs_common.cuh"
#include "rs_internal.h"

namespace rs {

// Shared-memory carve-up, in floats (every block 16-byte aligned).
struct ReplaySmem {
    int kv, vr, ar, sr, d1, d2, c1, c2, g1, g2, fw, gF, pre1, pre2, red, total;
};

__host__ __device__ inline int al4(int x) { return (x + 3) & ~3; }

__host__ __device__ inline ReplaySmem replay_smem(int HPC, int TMAX, int cap, int P, int N, int NW, int J) {
    ReplaySmem s;
    int o = 0;
    s.kv = o;   o += al4((cap + TMAX) * N);   // k_r (rows < cap) then q_i (rows cap + i), fp32
    s.vr = o;   o += al4(HPC * cap * P);      // record values: Mamba-2 x_r, GDN u_r (fp32)
    s.ar = o;   o += al4(HPC * cap);          // record decays alpha_r
    s.sr = o;   o += al4(HPC * cap);          // Mamba-2 record value scales dt_r
    s.d1 = o;   o += al4(cap * TMAX);         // Mamba-2 k_r.q_i ; GDN k_r.k_{m_i}
    s.d2 = o;   o += al4(cap * TMAX);         // GDN k_r.q_i
    s.c1 = o;   o += al4(HPC * TMAX * cap);   // replay coefficients (see phase 2)
    s.c2 = o;   o += al4(HPC * TMAX * cap);
    s.g1 = o;   o += al4(HPC * TMAX);         // checkpoint decays
    s.g2 = o;   o += al4(HPC * TMAX);
    s.fw = o;   o += al4(HPC * cap);          // fold weights
    s.gF = o;   o += al4(HPC);                // fold checkpoint decay
    s.pre1 = o; o += al4(HPC * TMAX * P);     // GDN committed-record replay terms
    s.pre2 = o; o += al4(HPC * TMAX * P);
    s.red = o;  o += al4(NW * HPC * (J > 0 ? J : 1) * P);
    s.total = o;
    return s;
}

// ---------------------------------------------------------------------------
// Everything after the pointer decision, for one checkpoint element type TE
// (float: the fp32 copy; uint16_t: the bf16 copy).
template <int KIND, int P, int N, int HPC, int TMAX, int NT, typename TE>
__device__ __forceinline__ void replay_body(const ReplayParams &p, float *sm, const ReplaySmem &S,
                                            const int b, const int h0, const int g, const int base,
                                            const int hc, const int T, const int F, const bool fold,
                                            const bool append) {
    using Gm = Geo<P, N, NT, TE>;
    constexpr int VEC = Gm::VEC, TPR = Gm::TPR, R = Gm::R;
    constexpr int JMAX = (KIND == RS_GDN ? 2 : 1) * TMAX;
    const int mode = p.mode;
    const int tid = threadIdx.x;
    const int pv = tid % TPR, n0 = (tid / TPR) * R, p0 = pv * VEC;
    const int H = p.H, G = p.G, cap = p.cap;
    const int J = (KIND == RS_GDN ? 2 : 1) * T;  // live vectors per head
    const int nrec = hc + T;  // records in the window after this launch's appends
    const size_t slab = (size_t)N * P;

    // ---- phase 1a: issue the checkpoint slab loads (consumed in phase 3 / 6)
    const TE *ck = sizeof(TE) == 4 ? reinterpret_cast<const TE *>(p.ckpt_hp)
                                   : reinterpret_cast<const TE *>(p.ckpt_lp);
    uint4 tile[HPC][R];
#pragma unroll
    for (int hd = 0; hd < HPC; ++hd) {
        const TE *src = ck + ((size_t)b * H + h0 + hd) * slab + (size_t)n0 * P + p0;
#pragma unroll
        for (int k = 0; k < R; ++k) tile[hd][k] = ld_stream(src + (size_t)k * P);
    }

    float *kv = sm + S.kv, *vr = sm + S.vr, *ar = sm + S.ar, *sr = sm + S.sr;
    auto slot = [&](int r) { return (base + r) % cap; };

    // ---- phase 1b: stage keys, queries, record values and decay inputs
    {
        // key rows r < nrec and query rows cap + i: 8 threads per row
        const int nrows = nrec + T;
        for (int rr = tid / 8; rr < nrows; rr += NT / 8) {
            const uint16_t *src;
            float *dst;
            if (rr < nrec) {
                dst = kv + (size_t)rr * N;
                if (rr < hc) {
                    src = p.buf_k + (((size_t)b * cap + slot(rr)) * G + g) * N;
                } else {
                    const int i = rr - hc;
                    src = (KIND == RS_MAMBA2 ? p.Bm : p.k) + (((size_t)b * T + i) * G + g) * N;
                }
            } else {
                const int i = rr - nrec;
                dst = kv + (size_t)(cap + i) * N;
                src = (KIND == RS_MAMBA2 ? p.Cm : p.q) + (((size_t)b * T + i) * G + g) * N;
            }
            bf16_row_to_smem(dst, src, N, tid % 8, 8);
        }
        // record values per head (Mamba-2: committed and new x; GDN: committed u)
        const int nv = KIND == RS_MAMBA2 ? nrec : hc;
        for (int it = tid; it < HPC * nv * (P / 4); it += NT) {
            const int c = it % (P / 4), r = (it / (P / 4)) % nv, hd = it / ((P / 4) * nv);
            const int hh = h0 + hd;
            float4 f;
            if (KIND == RS_MAMBA2) {
                const uint16_t *src = r < hc
                    ? static_cast<const uint16_t *>(p.buf_v) + (((size_t)b * cap + slot(r)) * H + hh) * P
                    : p.x + (((size_t)b * T + (r - hc)) * H + hh) * P;
                const uint2 u = *reinterpret_cast<const uint2 *>(src + 4 * c);
                f = make_float4(bf2f(u.x & 0xffffu), __uint_as_float(u.x & 0xffff0000u),
                                bf2f(u.y & 0xffffu), __uint_as_float(u.y & 0xffff0000u));
            } else {
                const float *src = static_cast<const float *>(p.buf_v) +
                                   (((size_t)b * cap + slot(r)) * H + hh) * P;
                f = reinterpret_cast<const float4 *>(src)[c];
            }
            reinterpret_cast<float4 *>(vr + ((size_t)hd * cap + r) * P)[c] = f;
        }
        // decays alpha_r (Mamba-2: exp(dt_r A_h), formed once when the record is
        // appended) and, for Mamba-2, the value scale dt_r (v_r = dt_r x_r)
        for (int it = tid; it < HPC * nrec; it += NT) {
            const int r = it % nrec, hd = it / nrec, hh = h0 + hd;
            float a, dtv = 0.f;
            if (r < hc) {
                const size_t rec = ((size_t)b * cap + slot(r)) * H + hh;
                a = p.buf_a[rec];
                if (KIND == RS_MAMBA2) dtv = p.buf_s[rec];
            } else {
                const size_t bti = ((size_t)b * T + (r - hc)) * H + hh;
                if (KIND == RS_MAMBA2) {
                    dtv = p.dt[bti];
                    a = expf(dtv * p.A[hh]);
                } else {
                    a = p.alpha[bti];
                }
                if (append) {
                    const size_t rec = ((size_t)b * cap + slot(r)) * H + hh;
                    p.buf_a[rec] = a;
                    if (KIND == RS_MAMBA2) p.buf_s[rec] = dtv;
                }
            }
            ar[hd * cap + r] = a;
            if (KIND == RS_MAMBA2) sr[hd * cap + r] = dtv;
        }
        // append this launch's keys and (Mamba-2) values; GDN u follows in phase 5
        if (append) {
            const bool first_of_group = (h0 % (H / G)) == 0;
            for (int it = tid; it < T * (N / 8); it += NT) {
                if (!first_of_group) break;
                const int i = it / (N / 8), c = it % (N / 8);
                const uint16_t *src = (KIND == RS_MAMBA2 ? p.Bm : p.k) + (((size_t)b * T + i) * G + g) * N;
                uint16_t *dst = p.buf_k + (((size_t)b * cap + slot(hc + i)) * G + g) * N;
                reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(src)[c];
            }
            if (KIND == RS_MAMBA2) {
                for (int it = tid; it < T * HPC * (P / 8); it += NT) {
                    const int c = it % (P / 8), hd = (it / (P / 8)) % HPC, i = it / ((P / 8) * HPC);
                    const int hh = h0 + hd;
                    const uint16_t *src = p.x + (((size_t)b * T + i) * H + hh) * P;
                    uint16_t *dst = static_cast<uint16_t *>(p.buf_v) + (((size_t)b * cap + slot(hc + i)) * H + hh) * P;
                    reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(src)[c];
                }
            }
        }
    }
    __syncthreads();

    // ---- phase 2a: key/query dot products of the head group (8 lanes per dot)
    float *d1 = sm + S.d1, *d2 = sm + S.d2;
    if (T > 0) {
        const int per = nrec * T;  // (r, i) pairs
        const int ndots = (KIND == RS_GDN ? 2 : 1) * per;
        for (int base_d = 0; base_d < ndots; base_d += NT / 8) {
            const int d = base_d + tid / 8, sub = tid % 8;
            float acc = 0.f;
            int r = 0, i = 0, which = 0;
            if (d < ndots) {
                which = d / per;
                r = (d % per) / T;
                i = d % T;
                const float *a = kv + (size_t)r * N;
                // Mamba-2: k_r . q_i ; GDN which 0: k_r . k_{hc+i}, which 1: k_r . q_i
                const float *bvec = (KIND == RS_GDN && which == 0) ? kv + (size_t)(hc + i) * N
                                                                   : kv + (size_t)(cap + i) * N;
                for (int n = sub * 4; n < N; n += 32) {
                    const float4 x4 = *reinterpret_cast<const float4 *>(a + n);
                    const float4 y4 = *reinterpret_cast<const float4 *>(bvec + n);
                    acc += x4.x * y4.x + x4.y * y4.y + x4.z * y4.z + x4.w * y4.w;
                }
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            if (d < ndots && sub == 0) (which == 0 ? d1 : d2)[r * TMAX + i] = acc;
        }
    }
    __syncthreads();

    // ---- phase 2b: decay coefficients per head
    // Record positions are 0-based; draft i sits at m_i = hc + i.  With
    // E(r, m) = prod_{s=r+1..m} alpha_s and gamma(m) = prod_{s<=m} alpha_s:
    //   Mamba-2  c1[i][r] = E(r, m_i) dt_r (k_r . q_i)   multiplies x_r[p] in y_i
    //            g1[i]    = gamma(m_i)
    //   GDN      c1[i][r] = E(r, m_i - 1) (k_r . k_{m_i})  (r < m_i)  -> S_{m_i - 1} k_{m_i}
    //            c2[i][r] = E(r, m_i) (k_r . q_i)          (r <= m_i) -> S_{m_i} q_i
    //            g1[i] = gamma(m_i - 1), g2[i] = gamma(m_i)
    //   fold of F records: fw[r] = E(r, F-1) (times dt_r for Mamba-2), gF = gamma(F-1)
    float *c1 = sm + S.c1, *c2 = sm + S.c2, *g1 = sm + S.g1, *g2 = sm + S.g2;
    float *fw = sm + S.fw, *gF = sm + S.gF;
    {
        const int nA = HPC * T * nrec;
        for (int it = tid; it < nA + HPC * T + HPC * F + HPC; it += NT) {
            if (it < nA) {
                const int r = it % nrec, i = (it / nrec) % T, hd = it / (nrec * T);
                const float *a = ar + hd * cap;
                const int m = hc + i;
                float e = 1.f;  // E(r, m - 1)
                for (int q = r + 1; q <= m - 1; ++q) e *= a[q];
                const float em = r == m ? 1.f : e * a[m];  // E(r, m)
                float v1 = 0.f, v2 = 0.f;
                if (KIND == RS_MAMBA2) {
                    if (r <= m) v1 = em * sr[hd * cap + r] * d1[r * TMAX + i];
                } else {
                    if (r < m) v1 = e * d1[r * TMAX + i];
                    if (r <= m) v2 = em * d2[r * TMAX + i];
                }
                c1[(hd * TMAX + i) * cap + r] = v1;
                c2[(hd * TMAX + i) * cap + r] = v2;
            } else if (it < nA + HPC * T) {
                const int j = it - nA, i = j % T, hd = j / T;
                const float *a = ar + hd * cap;
                const int m = hc + i;
                float e = 1.f;
                for (int q = 0; q < m; ++q) e *= a[q];
                if (KIND == RS_MAMBA2) {
                    g1[hd * TMAX + i] = e * a[m];
                } else {
                    g1[hd * TMAX + i] = e;          // gamma(m - 1)
                    g2[hd * TMAX + i] = e * a[m];   // gamma(m)
                }
            } else if (it < nA + HPC * T + HPC * F) {
                const int j = it - nA - HPC * T, r = j % F, hd = j / F;
                const float *a = ar + hd * cap;
                float e = 1.f;
                for (int q = r + 1; q < F; ++q) e *= a[q];
                fw[hd * cap + r] = KIND == RS_MAMBA2 ? e * sr[hd * cap + r] : e;
            } else {
                const int hd = it - nA - HPC * T - HPC * F;
                const float *a = ar + hd * cap;
                float e = 1.f;
                for (int q = 0; q < F; ++q) e *= a[q];
                gF[hd] = e;
            }
        }
    }
    __syncthreads();

    // ---- phase 2c (GDN): committed-record parts of S_{m_i-1} k_{m_i} and S_{m_i} q_i
    float *pre1 = sm + S.pre1, *pre2 = sm + S.pre2;
    if (KIND == RS_GDN && T > 0) {
        for (int it = tid; it < HPC * T * P; it += NT) {
            const int pp = it % P, i = (it / P) % T, hd = it / (P * T);
            float s1 = 0.f, s2 = 0.f;
            for (int r = 0; r < hc; ++r) {
                const float u = vr[((size_t)hd * cap + r) * P + pp];
                s1 += c1[(hd * TMAX + i) * cap + r] * u;
                s2 += c2[(hd * TMAX + i) * cap + r] * u;
            }
            pre1[(hd * TMAX + i) * P + pp] = s1;
            pre2[(hd * TMAX + i) * P + pp] = s2;
        }
    }

    // ---- phase 3: stream the checkpoint slab: acc[v] = S_c . vec_v over this thread's rows
    float *red = sm + S.red;
    if (T > 0) {
        float acc[HPC * JMAX][VEC];
#pragma unroll
        for (int a = 0; a < HPC * JMAX; ++a)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[a][e] = 0.f;
#pragma unroll
        for (int j = 0; j < JMAX; ++j) {
            if (j < J) {
                // Mamba-2: q_j ; GDN: j < T -> k_{hc+j}, else q_{j-T}
                const float *vec = kv + (size_t)((KIND == RS_GDN && j < T) ? hc + j
                                                 : cap + (KIND == RS_GDN ? j - T : j)) * N + n0;
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    const float w = vec[k];
#pragma unroll
                    for (int hd = 0; hd < HPC; ++hd) {
                        float s[VEC];
                        unpack<TE, VEC>(tile[hd][k], s);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[hd * JMAX + j][e] = fmaf(s[e], w, acc[hd * JMAX + j][e]);
                    }
                }
            }
        }
        // ---- phase 4: CTA reduction -> red[(hd * JMAX + j) * P + p]
        cta_reduce<NT, TPR, VEC, P, HPC * JMAX>(acc, HPC * JMAX, red);
    }

    // ---- phase 5: outputs and GDN correction terms, one thread per (head, value index)
    for (int it = tid; it < HPC * P; it += NT) {
        const int pp = it % P, hd = it / P, hh = h0 + hd;
        float *vrow = vr + (size_t)hd * cap * P + pp;  // vrow[r * P] = value of record r
        if (KIND == RS_MAMBA2) {
            const float Dh = p.D ? p.D[hh] : 0.f;
            for (int i = 0; i < T; ++i) {
                const int m = hc + i;
                float yv = g1[hd * TMAX + i] * red[((size_t)hd * JMAX + i) * P + pp];
                const float *cc = c1 + (hd * TMAX + i) * cap;
                for (int r = 0; r <= m; ++r) yv = fmaf(cc[r], vrow[(size_t)r * P], yv);
                yv = fmaf(Dh, vrow[(size_t)m * P], yv);
                p.y[(((size_t)b * T + i) * H + hh) * P + pp] = yv;
            }
        } else {
            float ud[TMAX];
#pragma unroll
            for (int i = 0; i < TMAX; ++i) {
                ud[i] = 0.f;
                if (i < T) {
                    const int m = hc + i;
                    const size_t bti = ((size_t)b * T + i) * H + hh;
                    float sk = g1[hd * TMAX + i] * red[((size_t)hd * JMAX + i) * P + pp] +
                               pre1[(hd * TMAX + i) * P + pp];
                    const float *cc1 = c1 + (hd * TMAX + i) * cap + hc;
#pragma unroll
                    for (int i2 = 0; i2 < TMAX; ++i2)
                        if (i2 < i) sk = fmaf(cc1[i2], ud[i2], sk);
                    const float u = p.beta[bti] * (bf2f(p.v[bti * P + pp]) - ar[hd * cap + m] * sk);
                    ud[i] = u;
                    vrow[(size_t)m * P] = u;
                    if (append)
                        static_cast<float *>(p.buf_v)[(((size_t)b * cap + slot(m)) * H + hh) * P + pp] = u;
                    float yv = g2[hd * TMAX + i] * red[((size_t)hd * JMAX + T + i) * P + pp] +
                               pre2[(hd * TMAX + i) * P + pp];
                    const float *cc2 = c2 + (hd * TMAX + i) * cap + hc;
#pragma unroll
                    for (int i2 = 0; i2 < TMAX; ++i2)
                        if (i2 <= i) yv = fmaf(cc2[i2], ud[i2], yv);
                    p.y[bti * P + pp] = yv;
                }
            }
        }
        // fold weights applied to the record values: vr[r] <- fw[r] * v_r
        for (int r = 0; r < F; ++r) vrow[(size_t)r * P] *= fw[hd * cap + r];
    }

    const bool materialize = mode == MODE_MATERIALIZE;
    if (!(fold || materialize)) return;
    __syncthreads();

    // ---- phase 6: S_new = gF * S_c + sum_{r<F} (fw_r v_r) k_r^T, from the registers
#pragma unroll
    for (int hd = 0; hd < HPC; ++hd) {
        const size_t off = ((size_t)b * H + h0 + hd) * slab + (size_t)n0 * P + p0;
        const float gf = gF[hd];
#pragma unroll
        for (int k = 0; k < R; ++k) {
            float s[VEC];
            unpack<TE, VEC>(tile[hd][k], s);
#pragma unroll
            for (int e = 0; e < VEC; ++e) s[e] *= gf;
            const int n = n0 + k;
            for (int r = 0; r < F; ++r) {
                const float kr = kv[(size_t)r * N + n];
                const float *cf = vr + ((size_t)hd * cap + r) * P + p0;
#pragma unroll
                for (int c = 0; c < VEC / 4; ++c) {
                    const float4 c4 = reinterpret_cast<const float4 *>(cf)[c];
                    s[4 * c + 0] = fmaf(c4.x, kr, s[4 * c + 0]);
                    s[4 * c + 1] = fmaf(c4.y, kr, s[4 * c + 1]);
                    s[4 * c + 2] = fmaf(c4.z, kr, s[4 * c + 2]);
                    s[4 * c + 3] = fmaf(c4.w, kr, s[4 * c + 3]);
                }
            }
            if (materialize) {
                store_f32<VEC>(p.out + off + (size_t)k * P, s);
            } else {
                if (p.ckpt_hp) store_f32<VEC>(p.ckpt_hp + off + (size_t)k * P, s);
                if (p.ckpt_lp) store_bf16<VEC>(p.ckpt_lp + off + (size_t)k * P, s);
            }
        }
    }
}

// ---------------------------------------------------------------------------
template <int KIND, int P, int N, int HPC, int TMAX, int NT>
__global__ void __launch_bounds__(NT) replay_kernel(const ReplayParams p) {
    extern __shared__ __align__(16) float sm[];
    const int b = blockIdx.y, h0 = blockIdx.x * HPC;
    const int g = h0 / (p.H / p.G);
    const int mode = p.mode, cap = p.cap, L = p.L;
    const int T = mode == MODE_DECODE ? 1 : (mode == MODE_VERIFY ? p.T : 0);
    const ReplaySmem S = replay_smem(HPC, TMAX, cap, P, N, NT / 32, (KIND == RS_GDN ? 2 : 1) * TMAX);

    const int base = p.base[b], hc = p.h[b], ndr = p.nd[b];
    int F = 0;
    bool fold = false, ok = true, append = false;
    unsigned err = 0;
    // a pointer state outside the buffer (never produced by the library) is
    // reported and the sequence left untouched rather than indexed with it
    const bool sane = base >= 0 && base < cap && hc >= 0 && hc <= cap && ndr >= 0 && ndr <= cap;
    if (!sane) {
        ok = false;
    } else if (mode == MODE_DECODE) {
        if (ndr) err |= RS_DEV_DRAFTS_PENDING;
        ok = hc + 1 <= cap;
        F = hc + 1;
        fold = F >= L;
        append = !fold;  // a folded record never needs its buffer slot
    } else if (mode == MODE_VERIFY) {
        if (ndr) err |= RS_DEV_DRAFTS_PENDING;
        ok = hc + T <= cap;
        fold = hc + T > L && hc > 0;
        F = fold ? hc : 0;
        append = true;
    } else {  // flush / materialize: the committed records
        F = hc;
        fold = mode == MODE_FLUSH && hc > 0;
    }
    if (!ok) err |= RS_DEV_CAPACITY;
    const bool work = ok && (mode != MODE_FLUSH || fold);
    if (work) {
        const bool lp = p.prec == RS_PREC_SHARED_BF16 ||
                        (p.prec == RS_PREC_TWO && !fold && mode != MODE_MATERIALIZE);
        if (lp)
            replay_body<KIND, P, N, HPC, TMAX, NT, uint16_t>(p, sm, S, b, h0, g, base, hc, T, F, fold, append);
        else
            replay_body<KIND, P, N, HPC, TMAX, NT, float>(p, sm, S, b, h0, g, base, hc, T, F, fold, append);
    }
    if (mode == MODE_MATERIALIZE) return;
    __syncthreads();
    if (threadIdx.x == 0) {
        if (err && h0 == 0) atomicOr(p.status, err);
        if (arrive_last(p.arrive + b, gridDim.x) && ok) {
            if (mode == MODE_DECODE) {
                if (fold) { p.base[b] = (base + F) % cap; p.h[b] = 0; }
                else p.h[b] = hc + 1;
                p.nd[b] = 0;
            } else if (mode == MODE_VERIFY) {
                if (fold) { p.base[b] = (base + hc) % cap; p.h[b] = 0; }
                p.nd[b] = T;
            } else if (fold) {  // flush
                p.base[b] = (base + hc) % cap;
                p.h[b] = 0;
            }
        }
    }
}

// ---------------------------------------------------------------------------
template <int KIND, int P, int N, int HPC, int TMAX, int NT>
static cudaError_t launch_replay(const ReplayParams &p, cudaStream_t stream) {
    // the reduction scratch holds JMAX vectors per head (see phase 4)
    const ReplaySmem S = replay_smem(HPC, TMAX, p.cap, P, N, NT / 32, (KIND == RS_GDN ? 2 : 1) * TMAX);
    const size_t smem = (size_t)S.total * sizeof(float);
    auto kern = replay_kernel<KIND, P, N, HPC, TMAX, NT>;
    static int smem_set = 0;  // largest opt-in already granted to this instantiation
    if ((int)smem > smem_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = (int)smem;
    }
    dim3 grid(p.H / HPC, p.B);
    kern<<<grid, NT, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int KIND, int P, int N, int NT>
static cudaError_t dispatch_T(const ReplayParams &p, int hpc, cudaStream_t s) {
    const int T = p.mode == MODE_VERIFY ? p.T : 1;
    if constexpr (KIND == RS_MAMBA2) {  // heads of a group share keys: two per CTA when possible
        if (T <= 1) return hpc == 2 ? launch_replay<KIND, P, N, 2, 1, NT>(p, s) : launch_replay<KIND, P, N, 1, 1, NT>(p, s);
        if (T <= 4) return hpc == 2 ? launch_replay<KIND, P, N, 2, 4, NT>(p, s) : launch_replay<KIND, P, N, 1, 4, NT>(p, s);
    } else {
        (void)hpc;
        if (T <= 1) return launch_replay<KIND, P, N, 1, 1, NT>(p, s);
        if (T <= 4) return launch_replay<KIND, P, N, 1, 4, NT>(p, s);
    }
    return launch_replay<KIND, P, N, 1, 8, NT>(p, s);
}

cudaError_t replay_launch(const ReplayParams &p, int kind, int P, int N, cudaStream_t s) {
    const int hpg = p.H / p.G;
    const int T = p.mode == MODE_VERIFY ? p.T : 1;
    if (kind == RS_MAMBA2) {
        const int hpc = (hpg % 2 == 0 && T <= 4) ? 2 : 1;
        if (P == 64 && N == 128) return dispatch_T<RS_MAMBA2, 64, 128, 256>(p, hpc, s);
        if (P == 64 && N == 64) return dispatch_T<RS_MAMBA2, 64, 64, 128>(p, hpc, s);
    } else {
        if (P == 128 && N == 128) return dispatch_T<RS_GDN, 128, 128, 256>(p, 1, s);
        if (P == 64 && N == 64) return dispatch_T<RS_GDN, 64, 64, 128>(p, 1, s);
    }
    return cudaErrorInvalidValue;
}

bool replay_shape_supported(int kind, int P, int N) {
    if (kind == RS_MAMBA2) return P == 64 && (N == 128 || N == 64);
    return (P == 128 && N == 128) || (P == 64 && N == 64);
}

}  // namespace rs
