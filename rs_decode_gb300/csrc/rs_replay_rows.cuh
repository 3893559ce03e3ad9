// Output-only replay kernels of the ReplaySSM decode path (Mamba-2 and Gated
// DeltaNet): standard decode with the flush route fused, speculative verify
// with the fold of committed records fused, forced flush, and materialise.
//
// The state of one (sequence, head) is S = gamma * S_c + sum_r w_r v_r k_r^T
// over the records r since the checkpoint S_c ("ReplaySSM: Cache SSM Inputs,
// Not State", section "How it works").  A step reads the checkpoint once and
// writes only outputs and the appended record; the checkpoint is rewritten
// only by a fold (the "flush route").
//
// Kernel structure: a persistent, warp-specialised streaming pipeline.
//   * Work unit = HU heads of one sequence that share one key group.
//   * A producer warp (one elected lane) plans each unit from the sequence's
//     pointers and streams the unit's checkpoint slabs (one per head, N x P,
//     contiguous; SPLIT row blocks per slab) into a ring of NS shared-memory
//     stages with bulk (TMA) copies that complete on mbarriers.  It runs
//     ahead into the next unit while the consumers finish the current one.
//   * NC consumer threads stage every small operand of the unit (buffered
//     records, the step's keys / queries / values, per-head constants) with
//     one batch of cp.async copies, compute the key.query dots and decay
//     coefficients once per unit, then per head: dot the slab with the query
//     (GDN: and key) vectors, reduce across warps, write the outputs (GDN:
//     and the correction term u), and on a fold rewrite the slab as
//     gamma S_c + (V diag(w)) K^T from the staged copy.  A stage is handed back
//     to the producer as soon as it has been read for the last time.
// Slabs are key-major ([N][P], value index contiguous): each consumer thread
// owns VEC value columns of R consecutive key rows, so its dot products
// accumulate locally and only a per-head cross-warp reduction is needed.
//
// Units are handed out dynamically (the launch's unit counter, rs_plan.cuh):
// the producer takes its CTA's next unit when it plans one and passes the
// unit's place to the consumers with the plan; an end plan (b = -1) ends them.
// Per-sequence pointers (base, h, nd) are read once per unit by the producer;
// the last unit to have read them (an arrival counter) writes the new values,
// so no second launch is needed.  Every wait is bounded: on a time-out the CTA
// raises RS_DEV_TIMEOUT, drains its copies and returns.
#pragma once

#include "rs_plan.cuh"

namespace rs {
namespace rows {

template <int KIND_, int P_, int N_, int HU_, int TMAX_, int NC_, int NS_, int SPLIT_>
struct PipeCfg {
    static constexpr int KIND = KIND_, P = P_, N = N_, HU = HU_, TMAX = TMAX_, NC = NC_, NS = NS_, SPLIT = SPLIT_;
    static constexpr int NCW = NC / 32;                   // consumer warps
    static constexpr int NT = NC + 32;                    // + one producer warp
    static constexpr int JMAX = (KIND == RS_GDN ? 2 : 1) * TMAX;
    static constexpr int NP = N / SPLIT;                  // key rows per stage
    static constexpr int STAGE = NP * P * 4;              // bytes of one fp32 row block = one stage
    static_assert(NS >= SPLIT, "a folding head keeps all its row blocks resident");
    // registers sized so that two CTAs fit on an SM (two-stage rings; the
    // draft-heavy T=8 shape excepted), three for the four-warp shapes of up to
    // 4 drafts (two for their 8-draft shape)
    static constexpr int MIN_BLOCKS = NC == 128 ? (TMAX <= 4 ? 3 : 2) : (NS <= 2 && TMAX <= 4) ? 2 : 1;
    // a folding unit converts its records' keys to fp32 once (single-query
    // launches: standard decode, flush, materialise); the draft buckets, whose
    // shared memory is fuller, convert key pairs as the fold reads them
    static constexpr bool KF = TMAX == 1;
};

// A unit's plan as the producer hands it to the consumers (b = -1: no more units).
struct RowPlan {
    SeqPlan s;
    int b, h0;
};

// Shared-memory carve-up, byte offsets (16-byte aligned; stages first).
struct PipeSmem {
    int stages, bars, plans, abort, kraw, xr, ar, sr, cst, vb, bt, d1, d2, c1, c2, g1, g2, fw, gF, pre1, pre2, red, kf,
        qf, total;
};

__host__ __device__ inline int al16(int x) { return (x + 15) & ~15; }

template <class C>
__host__ __device__ inline PipeSmem pipe_smem(int cap) {
    constexpr int HU = C::HU, TMAX = C::TMAX, P = C::P, N = C::N;
    constexpr bool GDN = C::KIND == RS_GDN;
    PipeSmem s;
    int o = 0;
    s.stages = o; o += C::NS * C::STAGE;
    s.bars = o;   o += al16((2 * C::NS + 4) * 8);
    s.plans = o;  o += al16(2 * (int)sizeof(RowPlan));
    s.abort = o;  o += 16;
    s.kf = o;     o += C::KF ? cap * N * 4 : 0;                     // folded records' keys, fp32 (just below kraw)
    s.kraw = o;   o += al16((cap + TMAX) * N * 2);                  // bf16 keys (rows < cap), queries (cap + i)
    s.xr = o;     o += al16(HU * cap * P * (GDN ? 4 : 2));          // Mamba-2 x bf16 / GDN u fp32 per record
    s.ar = o;     o += al16(HU * cap * 4);                          // decays alpha_r
    s.sr = o;     o += al16(HU * cap * 4);                          // Mamba-2 dt_r
    s.cst = o;    o += al16(2 * HU * 4);                            // Mamba-2 A_h, D_h
    s.vb = o;     o += GDN ? al16(TMAX * HU * P * 2) : 0;           // GDN drafts' v (bf16)
    s.bt = o;     o += GDN ? al16(TMAX * HU * 4) : 0;               // GDN drafts' beta
    s.d1 = o;     o += al16(cap * TMAX * 4);
    s.d2 = o;     o += al16(cap * TMAX * 4);
    s.c1 = o;     o += al16(HU * TMAX * cap * 4);
    s.c2 = o;     o += al16(HU * TMAX * cap * 4);
    s.g1 = o;     o += al16(HU * TMAX * 4);
    s.g2 = o;     o += al16(HU * TMAX * 4);
    s.fw = o;     o += al16(HU * cap * 4);
    s.gF = o;     o += al16(HU * 4);
    s.pre1 = o;   o += al16(HU * TMAX * P * 4);                     // record parts of the outputs
    s.pre2 = o;   o += GDN ? al16(HU * TMAX * P * 4) : 0;
    s.red = o;    o += al16(2 * C::NCW * C::JMAX * P * 4);          // double-buffered warp partials
    s.qf = o;     o += C::JMAX > 2 ? al16(N * C::JMAX * 4) : 0;     // draft buckets: dot vectors, fp32 [N][JMAX]
    s.total = o;
    return s;
}

// R consecutive bf16 values (16-byte aligned when R >= 8, 8-byte when R == 4) as fp32.
template <int R>
__device__ __forceinline__ void load_bf16_run(const uint16_t *src, float (&out)[R]) {
    if constexpr (R % 8 == 0) {
#pragma unroll
        for (int c = 0; c < R / 8; ++c) {
            float f[8];
            unpack<uint16_t, 8>(ld_u4(src + 8 * c), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) out[8 * c + e] = f[e];
        }
    } else if constexpr (R == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(src);
        out[0] = bf2f(u.x & 0xffffu); out[1] = __uint_as_float(u.x & 0xffff0000u);
        out[2] = bf2f(u.y & 0xffffu); out[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
#pragma unroll
        for (int k = 0; k < R; ++k) out[k] = bf2f(src[k]);
    }
}

// ---------------------------------------------------------------------------
// Producer: take each unit from the launch's counter, plan it, publish the
// plan, stream the unit's row blocks; then publish the end plan.
template <class C>
__device__ __forceinline__ void producer(const ReplayParams &p, uint8_t *sm, const PipeSmem &L, int units) {
    constexpr int HU = C::HU, NS = C::NS, N = C::N, P = C::P, SPLIT = C::SPLIT;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.bars), *empty = full + NS;
    uint64_t *pfull = empty + NS, *pempty = pfull + 2;
    RowPlan *plans = reinterpret_cast<RowPlan *>(sm + L.plans);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.abort);
    const unsigned upseq = p.H / HU;
    int it = 0, pu = 0;
    int u = next_unit(p);
    SeqPlan cur;
    if (u < units) {
        cur = plan_sequence(p, u / upseq);
        arrive_and_update(p, cur, u / upseq, upseq, (u % upseq) == 0);
    }
    bool stop = false;
    for (; u < units; ++pu) {
        const int b = u / upseq, h0 = (u % upseq) * HU;
        if (!wait_or_abort(pempty + (pu & 1), ((pu >> 1) & 1) ^ 1, abort_flag, p.status)) { stop = true; break; }
        plans[pu & 1].s = cur;
        plans[pu & 1].b = b;
        plans[pu & 1].h0 = h0;
        mbar_arrive(pfull + (pu & 1));  // release: the plan is visible to the consumers
        int un = units;
        SeqPlan next;
        bool planned = false;
        if (cur.work) {
            const bool lp = plan_reads_lp(p, cur);
            const unsigned slab = (unsigned)(N * P * (lp ? 2 : 4)), part = slab / SPLIT;
            const uint8_t *src = (lp ? reinterpret_cast<const uint8_t *>(p.ckpt_lp)
                                     : reinterpret_cast<const uint8_t *>(p.ckpt_hp)) +
                                 ((size_t)b * p.H + h0) * slab;
            for (int q = 0; q < HU * SPLIT; ++q, ++it) {
                const int st = it % NS;
                if (!wait_or_abort(empty + st, ((it / NS) & 1) ^ 1, abort_flag, p.status)) { stop = true; break; }
                mbar_arrive_expect_tx(full + st, part);
                bulk_copy_g2s(sm + L.stages + (size_t)st * C::STAGE, src + (size_t)q * part, part, full + st);
                if (q == 0) {  // plan the next unit while this one streams
                    un = next_unit(p);
                    if (un < units) {
                        next = plan_sequence(p, un / upseq);
                        arrive_and_update(p, next, un / upseq, upseq, (un % upseq) == 0);
                    }
                    planned = true;
                }
            }
            if (stop) break;
        }
        if (!planned) {
            un = next_unit(p);
            if (un < units) {
                next = plan_sequence(p, un / upseq);
                arrive_and_update(p, next, un / upseq, upseq, (un % upseq) == 0);
            }
        }
        u = un;
        cur = next;
    }
    if (!stop && wait_or_abort(pempty + (pu & 1), ((pu >> 1) & 1) ^ 1, abort_flag, p.status)) {
        plans[pu & 1].b = -1;  // the end plan
        mbar_arrive(pfull + (pu & 1));
    }
    planner_done(p, gridDim.x);
    if (*abort_flag) {
        // drain: wait (bounded) for the copies this thread may still have in flight
        for (int k = it - NS > 0 ? it - NS : 0; k < it; ++k) mbar_wait(full + k % NS, (k / NS) & 1);
    }
}

// ---------------------------------------------------------------------------
// Fold of one staged row block: S_new = gF S_c + sum_{r<F} (fw_r v_r) k_r^T,
// written to the checkpoint (both copies as present) or to the materialise
// output.  The thread's R rows are held as R/2 row pairs per column, so that
// one paired FMA (fma.rn.f32x2) applies a record to two rows: the record's
// keys for the rows are pairs as loaded (fp32 keys kf, or bf16 pairs widened
// with two integer operations), and the coefficient fw_r v_r of a column is
// formed once per record and broadcast into a pair.  The warp hands the stage
// back (one arrival on `empty`) as soon as its rows are in registers, so the
// next copy overlaps the fold's arithmetic and stores.
template <class C, typename TE, int R, int VEC>
__device__ __forceinline__ void fold_block(const ReplayParams &p, const TE *blk, uint64_t *empty, const uint16_t *kraw,
                                           const uint16_t *xb, const float *uf, const float *fw,
                                           float gf, int F, int cap, int j, int row0, int n0p, int p0, size_t goff,
                                           bool materialize) {
    constexpr int P = C::P, N = C::N, RP = R / 2;
    static_assert(R % 2 == 0, "rows are folded in pairs");
    unsigned long long o2[RP][VEC];
    {
        const unsigned long long g2 = f2_pack(gf, gf);
#pragma unroll
        for (int i = 0; i < RP; ++i) {
            float a[VEC], b[VEC];
            unpack<TE, VEC>(ld_u4(blk + (size_t)(n0p + 2 * i) * P + p0), a);
            unpack<TE, VEC>(ld_u4(blk + (size_t)(n0p + 2 * i + 1) * P + p0), b);
#pragma unroll
            for (int e = 0; e < VEC; ++e) o2[i][e] = f2_mul(f2_pack(a[e], b[e]), g2);
        }
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty);
    for (int r = 0; r < F; ++r) {
        float cf[VEC];
        const float w = fw[j * cap + r];
        if constexpr (C::KIND == RS_MAMBA2) {
            float xv[VEC];
            load_bf16_run<VEC>(xb + ((size_t)j * cap + r) * P + p0, xv);
#pragma unroll
            for (int e = 0; e < VEC; ++e) cf[e] = w * xv[e];
        } else {
#pragma unroll
            for (int e = 0; e < VEC; e += 4) {
                const float4 u4 = *reinterpret_cast<const float4 *>(uf + ((size_t)j * cap + r) * P + p0 + e);
                cf[e] = w * u4.x; cf[e + 1] = w * u4.y; cf[e + 2] = w * u4.z; cf[e + 3] = w * u4.w;
            }
        }
        unsigned long long kp[RP];
        if constexpr (C::KF) {  // the fp32 keys lie just below the bf16 ones
            // a pair of consecutive fp32 keys is one 64-bit word, the lower row low
            const unsigned long long *kr = reinterpret_cast<const unsigned long long *>(
                reinterpret_cast<const float *>(kraw) - (size_t)(cap - r) * N + row0 + n0p);
#pragma unroll
            for (int i = 0; i < RP; ++i) kp[i] = kr[i];
        } else {
            const uint32_t *kw = reinterpret_cast<const uint32_t *>(kraw + (size_t)r * N + row0 + n0p);
#pragma unroll
            for (int i = 0; i < RP; ++i) {
                const uint32_t u = kw[i];
                kp[i] = f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
            }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const unsigned long long cb = f2_pack(cf[e], cf[e]);
#pragma unroll
            for (int i = 0; i < RP; ++i) o2[i][e] = f2_fma(kp[i], cb, o2[i][e]);
        }
    }
#pragma unroll
    for (int i = 0; i < RP; ++i) {
        float a[VEC], b[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) f2_unpack(o2[i][e], a[e], b[e]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float(&o)[VEC] = h ? b : a;
            const size_t off = goff + (size_t)(row0 + n0p + 2 * i + h) * P + p0;
            if (materialize) {
                store_f32<VEC>(p.out + off, o);
            } else {
                if (p.ckpt_hp) store_f32<VEC>(p.ckpt_hp + off, o);
                if (p.ckpt_lp) store_bf16<VEC>(p.ckpt_lp + off, o);
            }
        }
    }
}

// Consumers: everything but the slab stream.
template <class C, typename TE>
__device__ __forceinline__ bool consume_unit(const ReplayParams &p, uint8_t *sm, const PipeSmem &L, const SeqPlan &s,
                                             const int b, const int h0, int &it) {
    constexpr int KIND = C::KIND, P = C::P, N = C::N, HU = C::HU, TMAX = C::TMAX, NC = C::NC, NS = C::NS;
    constexpr int JMAX = C::JMAX, NCW = C::NCW, SPLIT = C::SPLIT, NP = C::NP;
    using Gm = Geo<P, NP, NC, TE>;
    constexpr int VEC = Gm::VEC, TPR = Gm::TPR, R = Gm::R;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H, G = p.G, cap = p.cap, mode = p.mode;
    const int g = h0 / (H / G);
    const int n0p = (tid / TPR) * R, p0 = (tid % TPR) * VEC;  // rows within a row block, columns
    const int base = s.base, hc = s.hc, T = s.T, F = s.F;
    const bool fold = s.fold, append = s.append, materialize = mode == MODE_MATERIALIZE;
    const bool keep = fold || materialize;  // the staged slab is needed again after the reduction
    const int J = (KIND == RS_GDN ? 2 : 1) * T;
    const int nrec = hc + T;
    // buffer slot of record r: base < cap and r < cap for every planned unit
    // (plan_sequence), so one conditional subtract replaces the division
    auto slot = [&](int r) {
        const int v = base + r;
        return v >= cap ? v - cap : v;
    };

    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.bars), *empty = full + NS;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.abort);
    uint16_t *kraw = reinterpret_cast<uint16_t *>(sm + L.kraw);
    uint16_t *xb = reinterpret_cast<uint16_t *>(sm + L.xr);  // Mamba-2 x (bf16)
    float *uf = reinterpret_cast<float *>(sm + L.xr);        // GDN u (fp32)
    float *ar = reinterpret_cast<float *>(sm + L.ar), *sr = reinterpret_cast<float *>(sm + L.sr);
    float *cst = reinterpret_cast<float *>(sm + L.cst);      // A_h (HU), D_h (HU)
    uint16_t *vb = reinterpret_cast<uint16_t *>(sm + L.vb);
    float *bt = reinterpret_cast<float *>(sm + L.bt);
    float *d1 = reinterpret_cast<float *>(sm + L.d1), *d2 = reinterpret_cast<float *>(sm + L.d2);
    float *c1 = reinterpret_cast<float *>(sm + L.c1), *c2 = reinterpret_cast<float *>(sm + L.c2);
    float *g1 = reinterpret_cast<float *>(sm + L.g1), *g2 = reinterpret_cast<float *>(sm + L.g2);
    float *fw = reinterpret_cast<float *>(sm + L.fw), *gF = reinterpret_cast<float *>(sm + L.gF);
    float *pre1 = reinterpret_cast<float *>(sm + L.pre1), *pre2 = reinterpret_cast<float *>(sm + L.pre2);
    float *red = reinterpret_cast<float *>(sm + L.red);

    // ---- 1. one batch of cp.async copies for every small operand of the unit
    {
        constexpr int KC = N / 8;  // 16-byte chunks per key row
        for (int i2 = tid; i2 < (nrec + T) * KC; i2 += NC) {
            const int rr = i2 / KC, c = i2 % KC;
            const uint16_t *src;
            if (rr < hc) src = p.buf_k + (((size_t)b * cap + slot(rr)) * G + g) * N;
            else if (rr < nrec) src = (KIND == RS_MAMBA2 ? p.Bm : p.k) + (((size_t)b * T + (rr - hc)) * G + g) * N;
            else src = (KIND == RS_MAMBA2 ? p.Cm : p.q) + (((size_t)b * T + (rr - nrec)) * G + g) * N;
            const int row = rr < nrec ? rr : cap + (rr - nrec);
            cp_async16(kraw + (size_t)row * N + 8 * c, src + 8 * c);
        }
        if (KIND == RS_MAMBA2) {  // x of every record of the window, bf16
            constexpr int XC = P / 8;
            for (int i2 = tid; i2 < HU * nrec * XC; i2 += NC) {
                const int c = i2 % XC, r = (i2 / XC) % nrec, hd = i2 / (XC * nrec), hh = h0 + hd;
                const uint16_t *src = r < hc
                    ? static_cast<const uint16_t *>(p.buf_v) + (((size_t)b * cap + slot(r)) * H + hh) * P
                    : p.x + (((size_t)b * T + (r - hc)) * H + hh) * P;
                cp_async16(xb + ((size_t)hd * cap + r) * P + 8 * c, src + 8 * c);
            }
            // A (forms the new records' decays) and D (the skip term of the
            // outputs) only exist for launches that append records; flush and
            // materialise pass neither
            for (int i2 = tid; i2 < (T > 0 ? HU : 0); i2 += NC) {
                cp_async4(cst + i2, p.A + h0 + i2);
                if (p.D) cp_async4(cst + HU + i2, p.D + h0 + i2);
                else cst[HU + i2] = 0.f;
            }
        } else {  // committed u (fp32); the drafts' v (bf16) and beta
            constexpr int UC = P / 4, VC = P / 8;
            for (int i2 = tid; i2 < HU * hc * UC; i2 += NC) {
                const int c = i2 % UC, r = (i2 / UC) % hc, hd = i2 / (UC * hc), hh = h0 + hd;
                const float *src = static_cast<const float *>(p.buf_v) + (((size_t)b * cap + slot(r)) * H + hh) * P;
                cp_async16(uf + ((size_t)hd * cap + r) * P + 4 * c, src + 4 * c);
            }
            for (int i2 = tid; i2 < T * HU * VC; i2 += NC) {
                const int c = i2 % VC, hd = (i2 / VC) % HU, i = i2 / (VC * HU);
                cp_async16(vb + ((size_t)i * HU + hd) * P + 8 * c, p.v + (((size_t)b * T + i) * H + h0 + hd) * P + 8 * c);
            }
            for (int i2 = tid; i2 < T * HU; i2 += NC) {
                const int hd = i2 % HU, i = i2 / HU;
                cp_async4(bt + i2, p.beta + ((size_t)b * T + i) * H + h0 + hd);
            }
        }
        for (int i2 = tid; i2 < HU * nrec; i2 += NC) {  // decays and value scales
            const int r = i2 % nrec, hd = i2 / nrec, hh = h0 + hd;
            if (r < hc) {
                const size_t rec = ((size_t)b * cap + slot(r)) * H + hh;
                cp_async4(ar + hd * cap + r, p.buf_a + rec);
                if (KIND == RS_MAMBA2) cp_async4(sr + hd * cap + r, p.buf_s + rec);
            } else {
                const size_t bti = ((size_t)b * T + (r - hc)) * H + hh;
                if (KIND == RS_MAMBA2) cp_async4(sr + hd * cap + r, p.dt + bti);
                else cp_async4(ar + hd * cap + r, p.alpha + bti);
            }
        }
        cp_async_wait_all();
    }
    if (named_sync_or(1, NC, false)) return false;

    // ---- 2. the folded records' keys in fp32 (single-query configurations); the
    // dot vectors in fp32, key-major (draft buckets); new records' decays; appends
    if constexpr (JMAX > 2) {
        float *qf = reinterpret_cast<float *>(sm + L.qf);
        for (int i2 = tid; i2 < N * JMAX; i2 += NC) {
            const int jj = i2 % JMAX, n = i2 / JMAX;
            // Mamba-2: q_jj ; GDN: jj < T -> k_{hc+jj}, else q_{jj-T}
            const int row = (KIND == RS_GDN && jj < T) ? hc + jj : cap + (KIND == RS_GDN ? jj - T : jj);
            qf[i2] = jj < J ? bf2f(kraw[(size_t)row * N + n]) : 0.f;
        }
    }
    if constexpr (C::KF) {
        if (keep) {
            float *kf = reinterpret_cast<float *>(kraw) - (size_t)cap * N;
            for (int i2 = tid; i2 < F * (N / 8); i2 += NC) {
                const int r = i2 / (N / 8), c = i2 % (N / 8);
                float f[8];
                unpack<uint16_t, 8>(ld_u4(kraw + (size_t)r * N + 8 * c), f);
                float4 *d = reinterpret_cast<float4 *>(kf + (size_t)r * N + 8 * c);
                d[0] = make_float4(f[0], f[1], f[2], f[3]);
                d[1] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    }
    for (int i2 = tid; i2 < HU * T; i2 += NC) {
        const int i = i2 / HU, hd = i2 % HU, hh = h0 + hd, r = hc + i;
        float a;
        if (KIND == RS_MAMBA2) {  // alpha = exp(dt A), formed once when the record is appended
            a = expf(sr[hd * cap + r] * cst[hd]);
            ar[hd * cap + r] = a;
        } else {
            a = ar[hd * cap + r];
        }
        if (append) {
            const size_t rec = ((size_t)b * cap + slot(r)) * H + hh;
            p.buf_a[rec] = a;
            if (KIND == RS_MAMBA2) p.buf_s[rec] = sr[hd * cap + r];
        }
    }
    if (append) {
        if ((h0 % (H / G)) == 0) {  // the group's first unit appends the keys
            for (int i2 = tid; i2 < T * (N / 8); i2 += NC) {
                const int i = i2 / (N / 8), c = i2 % (N / 8);
                uint16_t *dst = p.buf_k + (((size_t)b * cap + slot(hc + i)) * G + g) * N;
                reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(kraw + (size_t)(hc + i) * N)[c];
            }
        }
        if (KIND == RS_MAMBA2) {
            for (int i2 = tid; i2 < T * HU * (P / 8); i2 += NC) {
                const int c = i2 % (P / 8), hd = (i2 / (P / 8)) % HU, i = i2 / ((P / 8) * HU);
                uint16_t *dst = static_cast<uint16_t *>(p.buf_v) + (((size_t)b * cap + slot(hc + i)) * H + h0 + hd) * P;
                reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(xb + ((size_t)hd * cap + hc + i) * P)[c];
            }
        }
    }

    // ---- 3. key/query dot products of the group (8 lanes per dot)
    if (T > 0) {
        const int per = nrec * T;
        const int ndots = (KIND == RS_GDN ? 2 : 1) * per;
        for (int bd = 0; bd < ndots; bd += NC / 8) {
            const int d = bd + tid / 8, sub = tid % 8;
            float acc = 0.f;
            int r = 0, i = 0, which = 0;
            if (d < ndots) {
                which = d / per;
                r = (d % per) / T;
                i = d % T;
                const uint16_t *a = kraw + (size_t)r * N;
                // Mamba-2: k_r . q_i ; GDN which 0: k_r . k_{hc+i}, which 1: k_r . q_i
                const uint16_t *bv = (KIND == RS_GDN && which == 0) ? kraw + (size_t)(hc + i) * N
                                                                    : kraw + (size_t)(cap + i) * N;
                for (int n = sub * 8; n < N; n += 64) {
                    float fa[8], fb[8];
                    unpack<uint16_t, 8>(ld_u4(a + n), fa);
                    unpack<uint16_t, 8>(ld_u4(bv + n), fb);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc = fmaf(fa[e], fb[e], acc);
                }
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            if (d < ndots && sub == 0) (which == 0 ? d1 : d2)[r * TMAX + i] = acc;
        }
    }
    if (named_sync_or(1, NC, false)) return false;

    // ---- 4. decay coefficients per head
    // Record positions are 0-based; draft i sits at m_i = hc + i.  With
    // E(r, m) = prod_{s=r+1..m} alpha_s and gamma(m) = prod_{s<=m} alpha_s:
    //   Mamba-2  c1[i][r] = E(r, m_i) dt_r (k_r . q_i)   multiplies x_r[p] in y_i;  g1[i] = gamma(m_i)
    //   GDN      c1[i][r] = E(r, m_i - 1) (k_r . k_{m_i})  (r < m_i)  -> S_{m_i - 1} k_{m_i}
    //            c2[i][r] = E(r, m_i) (k_r . q_i)          (r <= m_i) -> S_{m_i} q_i
    //            g1[i] = gamma(m_i - 1), g2[i] = gamma(m_i)
    //   fold of F records: fw[r] = E(r, F-1) (times dt_r for Mamba-2), gF = gamma(F-1)
    // One warp per head, one lane per record: a reverse product scan of
    // v_s = (s < hc ? alpha_s : 1) gives E(r, hc-1) in lane r and gamma(hc-1)
    // in lane 0; each further bound m (up to hc+T-1; F-1 is among them) takes
    // one more factor: E(r, m) = E(r, m-1) alpha_m for r < m, E(m, m) = 1.
    for (int hd = warp; hd < HU; hd += NCW) {
        const float al = lane < nrec ? ar[hd * cap + lane] : 1.f;
        const float dtr = KIND == RS_MAMBA2 && lane < nrec ? sr[hd * cap + lane] : 1.f;
        float inc = lane < hc ? al : 1.f;  // inclusive: prod_{s >= lane} v_s
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_down_sync(0xffffffffu, inc, off);
            if (lane + off < 32) inc *= o;
        }
        float E = __shfl_down_sync(0xffffffffu, inc, 1);  // prod_{s > lane} v_s = E(lane, hc-1)
        if (lane == 31) E = 1.f;
        float gam = __shfl_sync(0xffffffffu, inc, 0);  // gamma(hc-1)
        for (int m = hc - 1; m < hc + T; ++m) {
            if (m >= hc) {
                const float am = __shfl_sync(0xffffffffu, al, m);  // alpha_m (m < nrec <= 32)
                E = lane < m ? E * am : 1.f;
                gam *= am;
            }
            const int i = m - hc;  // the draft whose own position is m (-1: none)
            if (lane < nrec) {
                if (KIND == RS_MAMBA2) {
                    if (i >= 0) c1[(hd * TMAX + i) * cap + lane] = lane <= m ? E * dtr * d1[lane * TMAX + i] : 0.f;
                } else {
                    if (i >= 0) c2[(hd * TMAX + i) * cap + lane] = lane <= m ? E * d2[lane * TMAX + i] : 0.f;
                    if (i + 1 < T) c1[(hd * TMAX + i + 1) * cap + lane] = lane <= m ? E * d1[lane * TMAX + i + 1] : 0.f;
                }
                if (m == F - 1 && lane < F) fw[hd * cap + lane] = KIND == RS_MAMBA2 ? E * dtr : E;
            }
            if (lane == 0) {
                if (i >= 0) {
                    if (KIND == RS_MAMBA2) g1[hd * TMAX + i] = gam;
                    else g2[hd * TMAX + i] = gam;
                }
                if (KIND == RS_GDN && i + 1 < T) g1[hd * TMAX + i + 1] = gam;
                if (m == F - 1) gF[hd] = gam;
            }
        }
        if (F == 0 && lane == 0) gF[hd] = 1.f;
    }
    if (named_sync_or(1, NC, false)) return false;

    // ---- 5 (Mamba-2): record parts of the outputs, rec_i[p] = sum_{r <= m_i} c1[i][r] x_r[p]
    // + D x_{m_i}[p]; one task per head and 4 columns, all drafts at once
    if (KIND == RS_MAMBA2 && T > 0) {
        constexpr int PC = P / 4;
        for (int i2 = tid; i2 < HU * PC; i2 += NC) {
            const int pc = i2 % PC, hd = i2 / PC;
            const float d = cst[HU + hd];
            float a[TMAX][4];
#pragma unroll
            for (int i = 0; i < TMAX; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) a[i][e] = 0.f;
            const uint16_t *xr = xb + (size_t)hd * cap * P + 4 * pc;
            for (int r = 0; r < nrec; ++r) {
                float xv[4];
                load_bf16_run<4>(xr + (size_t)r * P, xv);
#pragma unroll
                for (int i = 0; i < TMAX; ++i) {
                    if (i < T && r <= hc + i) {
                        const float c = c1[(hd * TMAX + i) * cap + r] + (r == hc + i ? d : 0.f);
#pragma unroll
                        for (int e = 0; e < 4; ++e) a[i][e] = fmaf(c, xv[e], a[i][e]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < TMAX; ++i)
                if (i < T)
                    *reinterpret_cast<float4 *>(pre1 + (hd * TMAX + i) * P + 4 * pc) =
                        make_float4(a[i][0], a[i][1], a[i][2], a[i][3]);
        }
        // read after the first head's partial barrier
    }

    // ---- 5 (GDN): committed-record parts of S_{m_i-1} k_{m_i} and S_{m_i} q_i
    if (KIND == RS_GDN && T > 0) {
        for (int i2 = tid; i2 < HU * T * P; i2 += NC) {
            const int pp = i2 % P, i = (i2 / P) % T, hd = i2 / (P * T);
            float s1 = 0.f, s2 = 0.f;
            for (int r = 0; r < hc; ++r) {
                const float u = uf[((size_t)hd * cap + r) * P + pp];
                s1 = fmaf(c1[(hd * TMAX + i) * cap + r], u, s1);
                s2 = fmaf(c2[(hd * TMAX + i) * cap + r], u, s2);
            }
            pre1[(hd * TMAX + i) * P + pp] = s1;
            pre2[(hd * TMAX + i) * P + pp] = s2;
        }
        // read after the first head's partial barrier
    }

    // ---- 6. the unit's heads: SPLIT ring stages each
    for (int j = 0; j < HU; ++j) {
        const int hh = h0 + j, it0 = it;
        const size_t goff = ((size_t)b * H + hh) * ((size_t)N * P);
        float acc[JMAX][VEC];
#pragma unroll
        for (int a = 0; a < JMAX; ++a)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[a][e] = 0.f;
        unsigned long long acc2[JMAX > 2 ? JMAX / 2 : 1][VEC];  // draft buckets: vector pairs per column
#pragma unroll
        for (int m = 0; m < (JMAX > 2 ? JMAX / 2 : 1); ++m)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc2[m][e] = 0ull;
        bool ok = true;
        for (int part = 0; part < SPLIT; ++part, ++it) {
            const int st = it % NS;
            ok = wait_or_abort(full + st, (it / NS) & 1, abort_flag, p.status) && ok;
            const TE *blk = reinterpret_cast<const TE *>(sm + L.stages + (size_t)st * C::STAGE);
            if (ok && J > 0) {
                const int row0 = part * NP + n0p;
                if constexpr (JMAX <= 2) {
                    // the dot vectors' bf16 values at the thread's R consecutive
                    // rows: one vector load per vector, kept packed (two values
                    // per register) and unpacked where used
                    static_assert(R == 2 || R == 4 || R == 8, "rows per thread");
                    uint32_t wv[JMAX][R / 2];
#pragma unroll
                    for (int jj = 0; jj < JMAX; ++jj) {
                        if (jj < J) {
                            // Mamba-2: q_jj ; GDN: jj < T -> k_{hc+jj}, else q_{jj-T}
                            const int row =
                                (KIND == RS_GDN && jj < T) ? hc + jj : cap + (KIND == RS_GDN ? jj - T : jj);
                            const uint16_t *src = kraw + (size_t)row * N + row0;
                            if constexpr (R == 8) {
                                const uint4 u = ld_u4(src);
                                wv[jj][0] = u.x; wv[jj][1] = u.y; wv[jj][2] = u.z; wv[jj][3] = u.w;
                            } else if constexpr (R == 4) {
                                const uint2 u = *reinterpret_cast<const uint2 *>(src);
                                wv[jj][0] = u.x; wv[jj][1] = u.y;
                            } else {
                                wv[jj][0] = *reinterpret_cast<const uint32_t *>(src);
                            }
                        }
                    }
#pragma unroll
                    for (int k = 0; k < R; ++k) {
                        float sv[VEC];
                        unpack<TE, VEC>(ld_u4(blk + (size_t)(n0p + k) * P + p0), sv);
#pragma unroll
                        for (int jj = 0; jj < JMAX; ++jj) {
                            if (jj < J) {
                                const uint32_t pr = wv[jj][k >> 1];
                                const float w =
                                    (k & 1) ? __uint_as_float(pr & 0xffff0000u) : __uint_as_float(pr << 16);
#pragma unroll
                                for (int e = 0; e < VEC; ++e) acc[jj][e] = fmaf(sv[e], w, acc[jj][e]);
                            }
                        }
                    }
                } else {
                    // more vectors (draft buckets): a row's vector values are
                    // one fp32 run of qf, consecutive vectors pairing up, and
                    // each slab value is broadcast into a pair, so that one
                    // paired FMA serves two vectors
                    const float *qf = reinterpret_cast<const float *>(sm + L.qf);
#pragma unroll
                    for (int k = 0; k < R; ++k) {
                        float sv[VEC];
                        unpack<TE, VEC>(ld_u4(blk + (size_t)(n0p + k) * P + p0), sv);
                        const unsigned long long *wq =
                            reinterpret_cast<const unsigned long long *>(qf + (size_t)(row0 + k) * JMAX);
                        unsigned long long w2[JMAX / 2];
#pragma unroll
                        for (int m = 0; m < JMAX / 2; ++m) w2[m] = wq[m];
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const unsigned long long sb = f2_pack(sv[e], sv[e]);
#pragma unroll
                            for (int m = 0; m < JMAX / 2; ++m) acc2[m][e] = f2_fma(w2[m], sb, acc2[m][e]);
                        }
                    }
                }
            }
            if (!keep) {  // last read of this row block: hand the stage back
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + st);
            }
        }
        if constexpr (JMAX > 2) {
#pragma unroll
            for (int m = 0; m < JMAX / 2; ++m)
#pragma unroll
                for (int e = 0; e < VEC; ++e) f2_unpack(acc2[m][e], acc[2 * m][e], acc[2 * m + 1][e]);
        }
        // intra-warp reduction over the row groups of the warp, then per-warp partials
#pragma unroll
        for (int off = TPR; off < 32; off <<= 1)
#pragma unroll
            for (int a = 0; a < JMAX; ++a)
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[a][e] += __shfl_xor_sync(0xffffffffu, acc[a][e], off);
        float *rb = red + (size_t)(j & 1) * NCW * JMAX * P;
        if (lane < TPR) {
#pragma unroll
            for (int a = 0; a < JMAX; ++a)
                if (a < J)
#pragma unroll
                    for (int c = 0; c < VEC / 4; ++c)
                        reinterpret_cast<float4 *>(rb + ((size_t)warp * JMAX + a) * P + p0)[c] =
                            make_float4(acc[a][4 * c], acc[a][4 * c + 1], acc[a][4 * c + 2], acc[a][4 * c + 3]);
        }

        if (KIND == RS_MAMBA2 && keep && ok) {  // the Mamba-2 fold needs nothing the reduction produces
            for (int part = 0; part < SPLIT; ++part) {
                const int st = (it0 + part) % NS;
                fold_block<C, TE, R, VEC>(p, reinterpret_cast<const TE *>(sm + L.stages + (size_t)st * C::STAGE),
                                          empty + st, kraw, xb, uf, fw, gF[j], F, cap, j, part * NP, n0p, p0, goff,
                                          materialize);
            }
        }
        if (named_sync_or(1, NC, !ok)) return false;  // partials of head j complete

        if (KIND == RS_MAMBA2) {
            // y_i[p] = gamma(m_i) (S_c q_i)[p] + rec_i[p]
            for (int i2 = tid; i2 < T * P; i2 += NC) {
                const int i = i2 / P, pp = i2 % P;
                float sq = 0.f;
#pragma unroll
                for (int w = 0; w < NCW; ++w) sq += rb[((size_t)w * JMAX + i) * P + pp];
                p.y[(((size_t)b * T + i) * H + hh) * P + pp] = fmaf(g1[j * TMAX + i], sq, pre1[(j * TMAX + i) * P + pp]);
            }
        } else {
            // GDN: per value index, the recurrence over the drafts
            for (int pp = tid; pp < P; pp += NC) {
                float ud[TMAX];
#pragma unroll
                for (int i = 0; i < TMAX; ++i) {
                    ud[i] = 0.f;
                    if (i < T) {
                        const int m = hc + i;
                        float ak = 0.f, bq = 0.f;  // (S_c k_{m_i})[p], (S_c q_i)[p]
#pragma unroll
                        for (int w = 0; w < NCW; ++w) {
                            ak += rb[((size_t)w * JMAX + i) * P + pp];
                            bq += rb[((size_t)w * JMAX + T + i) * P + pp];
                        }
                        float sk = g1[j * TMAX + i] * ak + pre1[(j * TMAX + i) * P + pp];
                        const float *cc1 = c1 + (j * TMAX + i) * cap + hc;
#pragma unroll
                        for (int i3 = 0; i3 < TMAX; ++i3)
                            if (i3 < i) sk = fmaf(cc1[i3], ud[i3], sk);
                        const float u = bt[i * HU + j] * (bf2f(vb[((size_t)i * HU + j) * P + pp]) - ar[j * cap + m] * sk);
                        ud[i] = u;
                        uf[((size_t)j * cap + m) * P + pp] = u;
                        if (append) static_cast<float *>(p.buf_v)[(((size_t)b * cap + slot(m)) * H + hh) * P + pp] = u;
                        float yv = g2[j * TMAX + i] * bq + pre2[(j * TMAX + i) * P + pp];
                        const float *cc2 = c2 + (j * TMAX + i) * cap + hc;
#pragma unroll
                        for (int i3 = 0; i3 < TMAX; ++i3)
                            if (i3 <= i) yv = fmaf(cc2[i3], ud[i3], yv);
                        p.y[(((size_t)b * T + i) * H + hh) * P + pp] = yv;
                    }
                }
            }
            if (keep) {
                if (named_sync_or(1, NC, false)) return false;  // the new record's u is in uf
                for (int part = 0; part < SPLIT; ++part) {
                    const int st = (it0 + part) % NS;
                    fold_block<C, TE, R, VEC>(p, reinterpret_cast<const TE *>(sm + L.stages + (size_t)st * C::STAGE),
                                              empty + st, kraw, xb, uf, fw, gF[j], F, cap, j, part * NP, n0p, p0,
                                              goff, materialize);
                }
            }
        }
    }
    // the next unit's staging overwrites shared operands still read above
    return !named_sync_or(1, NC, false);
}

template <class C>
__device__ __forceinline__ void consumer(const ReplayParams &p, uint8_t *sm, const PipeSmem &L) {
    uint64_t *pfull = reinterpret_cast<uint64_t *>(sm + L.bars) + 2 * C::NS, *pempty = pfull + 2;
    const RowPlan *plans = reinterpret_cast<const RowPlan *>(sm + L.plans);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.abort);
    int it = 0;
    for (int pu = 0;; ++pu) {
        const bool ok = wait_or_abort(pfull + (pu & 1), (pu >> 1) & 1, abort_flag, p.status);
        RowPlan rp;
        if (ok) rp = plans[pu & 1];
        if (named_sync_or(1, C::NC, !ok)) return;
        if (threadIdx.x == 0) mbar_arrive(pempty + (pu & 1));
        if (rp.b < 0) return;  // the end plan
        if (!rp.s.work) continue;
        const bool done = plan_reads_lp(p, rp.s) ? consume_unit<C, uint16_t>(p, sm, L, rp.s, rp.b, rp.h0, it)
                                                 : consume_unit<C, float>(p, sm, L, rp.s, rp.b, rp.h0, it);
        if (!done) return;
    }
}

template <class C>
__global__ void __launch_bounds__(C::NT, C::MIN_BLOCKS) replay_pipe_kernel(const ReplayParams p, int units) {
    extern __shared__ __align__(128) uint8_t sm[];
    const PipeSmem L = pipe_smem<C>(p.cap);
    if (threadIdx.x == 0) {
        uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bars);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bars + s, 1);                 // full: the producer's expect_tx arrival
            mbar_init(bars + C::NS + s, C::NCW);    // empty: one arrival per consumer warp
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(bars + 2 * C::NS + k, 1);     // plan full
            mbar_init(bars + 2 * C::NS + 2 + k, 1); // plan empty
        }
        *reinterpret_cast<volatile int *>(sm + L.abort) = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= C::NC) {
        if (threadIdx.x == C::NC) producer<C>(p, sm, L, units);
        return;
    }
    consumer<C>(p, sm, L);
}

// ---------------------------------------------------------------------------
template <class C>
cudaError_t launch_pipe(const ReplayParams &p, cudaStream_t stream) {
    const PipeSmem L = pipe_smem<C>(p.cap);
    const int smem = L.total;
    auto kern = replay_pipe_kernel<C>;
    static SmemGrants grants;  // this instantiation's opt-in, per device
    cudaError_t e = grant_smem(reinterpret_cast<const void *>(kern), smem, grants);
    if (e != cudaSuccess) return e;
    int per_sm = 0, dev = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::NT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int units = p.B * (p.H / C::HU);
    const int grid = units < sms * per_sm ? units : sms * per_sm;
    kern<<<grid, C::NT, smem, stream>>>(p, units);
    return cudaGetLastError();
}

// Launch shapes, tried in order: (four-warp configurations of up to 4 drafts)
// three CTAs per SM; two CTAs per SM with a two-stage ring (one CTA's per-unit
// and per-head serial phases overlap the other's streaming); else one CTA per
// SM with a deeper ring that covers those phases itself; else one CTA with two
// stages.  Within a tier, the most heads per unit whose count divides the group
// and whose shared memory fits.
constexpr int kMaxSmemPerBlock = 227 * 1024;
constexpr int kTwoPerSm = kMaxSmemPerBlock / 2 - 1024;
constexpr int kThreePerSm = kMaxSmemPerBlock / 3 - 1024;

template <class C>
bool try_shape(const ReplayParams &p, int hpg, int limit, cudaStream_t s, cudaError_t &err) {
    if (hpg % C::HU != 0 || pipe_smem<C>(p.cap).total > limit) return false;
    err = launch_pipe<C>(p, s);
    return true;
}

template <int KIND, int P, int N, int NC, int TMAX, int SPLIT, int... HUS>
cudaError_t launch_shape(const ReplayParams &p, cudaStream_t s) {
    const int hpg = p.H / p.G;
    cudaError_t e = cudaErrorInvalidValue;
    constexpr int DEEP = 4;
    if constexpr (NC == 128 && TMAX <= 4)
        if ((try_shape<PipeCfg<KIND, P, N, HUS, TMAX, NC, 2, SPLIT>>(p, hpg, kThreePerSm, s, e) || ...)) return e;
    if ((try_shape<PipeCfg<KIND, P, N, HUS, TMAX, NC, 2, SPLIT>>(p, hpg, kTwoPerSm, s, e) || ...)) return e;
    if constexpr (TMAX == 8) {
        // one CTA per SM (buffers too large for two): the 8-draft bucket
        // prefers more heads per unit with three stages to fewer with four (8
        // consumer warps, B = 256, 8 drafts: 8 heads and 3 stages 0.616 ms per
        // round, 4 heads and 4 stages 0.837 ms)
        if (((try_shape<PipeCfg<KIND, P, N, HUS, TMAX, NC, DEEP, SPLIT>>(p, hpg, kMaxSmemPerBlock, s, e) ||
              try_shape<PipeCfg<KIND, P, N, HUS, TMAX, NC, 3, SPLIT>>(p, hpg, kMaxSmemPerBlock, s, e)) || ...))
            return e;
    }
    if ((try_shape<PipeCfg<KIND, P, N, HUS, TMAX, NC, DEEP, SPLIT>>(p, hpg, kMaxSmemPerBlock, s, e) || ...)) return e;
    if ((try_shape<PipeCfg<KIND, P, N, HUS, TMAX, NC, 2, SPLIT>>(p, hpg, kMaxSmemPerBlock, s, e) || ...)) return e;
    return cudaErrorInvalidConfiguration;
}

// Verify launches instantiate the draft-count buckets 1, 4 and 8.
template <int KIND, int P, int N, int NC, int SPLIT, int... HUS>
cudaError_t dispatch_shape(const ReplayParams &p, cudaStream_t s) {
    const int T = p.mode == MODE_VERIFY ? p.T : 1;
    if (T <= 1) return launch_shape<KIND, P, N, NC, 1, SPLIT, HUS...>(p, s);
    if (T <= 4) return launch_shape<KIND, P, N, NC, 4, SPLIT, HUS...>(p, s);
    return launch_shape<KIND, P, N, NC, 8, SPLIT, HUS...>(p, s);
}

}  // namespace rows
}  // namespace rs
