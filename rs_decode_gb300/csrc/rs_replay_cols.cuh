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
// Kernel structure: a persistent, warp-specialised pipeline with three roles.
//   * Work unit = HU heads of one sequence that share one key group.
//   * A producer warp: one lane plans units ahead (reads a sequence's
//     pointers, takes part in the pointer update) and ends the pipeline with
//     an end plan; another streams each unit's checkpoint slabs, once the prep
//     warps have taken up its plan, into a ring of NS shared-memory stages
//     with tiled tensor copies (TMA) that complete on mbarriers.  A stage is
//     one row block of a slab: 16 KiB of whole key rows (contiguous in HBM),
//     stored with the 128-byte swizzle, so a slab takes P*sizeof(elem)/128
//     stages.  (Tensor-core launches stream the bf16 copy in column blocks
//     instead; see the TC instantiation below.)
//   * Three prep warps build each unit's context one unit ahead of the
//     consumers, in a double buffer: they
//     stage every small operand (buffered records, the step's keys / queries
//     / values, per-head constants) with cp.async, append the new records, and
//     compute the key.query dots, the decay coefficients (product scans over
//     the records), the fp32 dot vectors and the record parts of the outputs.
//   * Four consumer warps only stream the heads.  Per head each warp works
//     alone on its own value columns: it dots them with the query (GDN: key
//     and query) vectors over every row block, reduces over its lanes with
//     shuffles, writes the outputs (GDN: runs the recurrence over the drafts
//     that gives the correction u), and on a fold rewrites its columns as
//     gamma S_c + (V diag(w)) K^T from the staged copy.  No barrier spans the
//     consumer warps; a stage goes back to the producer once every consumer
//     warp has read it, a context once every consumer warp is done with it.
// Slabs are key-major ([N][P], value index contiguous).  A stage holds its rows
// as 128-byte lines (row-major, NCB lines per row); 16-byte chunk c of line l
// sits at l*128 + ((c ^ (l & 7)) << 4).  Each shared-memory phase of 8 lanes
// reads chunks that land in 8 different bank groups (see WGeo).
//
// Per-sequence pointers (base, h, nd) are read once per unit by the planner;
// the last unit to have read them (an arrival counter) writes the new values,
// so no second launch is needed.  Every wait is bounded: on a time-out the CTA
// raises RS_DEV_TIMEOUT, drains its copies and returns.
//
// Per-channel decay (RS_KDA, a reading of Kimi Delta Attention: GDN with one
// decay per key channel) runs the GDN structure with three changes: the prep
// warps form per-channel suffix products of the decays in one reverse scan per
// head and fold them into the record dots and the fold keys; the dot vectors
// are per head, gamma (.) k and gamma (.) q, so the consumers' dots need no
// decay factor; and the fold scales each key row n of the slab by gamma[n].
//
// Two instantiations per shape.  TC = false: CUDA cores only, two CTAs per SM.
// TC = true (two-precision GDN launches): the bf16 blocks are dotted with the
// draft vectors on the tensor cores (tcgen05.mma, accumulator in TMEM).  A
// kernel that allocates tensor memory is resident one CTA per SM, so the TC
// instantiation runs two pipelines side by side in one CTA.
#pragma once

#include <cuda.h>
#include <string.h>

#include "rs_plan.cuh"

namespace rs {
namespace cols {

// Compile-time shape of one kernel instantiation: family, slab shape and the
// draft-count bucket.  Heads per unit (HU) and ring depth (NS) are launch
// arguments.
template <int KIND_, int P_, int N_, int TMAX_>
struct RCfg {
    static constexpr int KIND = KIND_, P = P_, N = N_, TMAX = TMAX_;
    static constexpr bool DELTA = KIND != RS_MAMBA2;    // records hold the correction u (GDN, KDA)
    static constexpr bool KDA = KIND == RS_KDA;          // one decay per key channel
    static constexpr int NCW = 4;                         // consumer warps (warps 0..NCW-1)
    static constexpr int NPW = 3;                         // prep warps (after the producer warp)
    static constexpr int NT = 32 * (NCW + 1 + NPW);       // + the producer warp (warp NCW)
    static constexpr int PREP0 = 32 * (NCW + 1);          // first prep thread
    static constexpr int NPT = 32 * NPW;                  // prep threads
    // vectors dotted with every slab: Mamba-2 the queries C_i; GDN the keys
    // k_{m_i} (slots 0..TMAX-1) and the queries q_i (slots TMAX..2TMAX-1);
    // KDA the same scaled per head by the channels' decay products
    static constexpr int JP = (DELTA ? 2 : 1) * TMAX;
    static constexpr int STAGE = N * 128;                 // one row block: N lines of 128 bytes
    static constexpr int QW = JP % 4 == 0 ? 4 : (JP % 2 == 0 ? 2 : 1);  // query floats per shared-memory vector
    static constexpr int QC = JP / QW;                    // vectors per key row
    static constexpr int MIN_BLOCKS = 2;                  // two CTAs per SM
    // dot vectors per pass over a staged head: at most 64 partial sums per lane
    template <int VEC> static constexpr int jn() { return VEC * JP <= 64 ? JP : 64 / VEC; }
    static_assert(N % 8 == 0 && N <= 256, "a stage is one tensor box");
    // the Mamba-2 output reduction halves down to single sums: a power-of-two bucket
    static_assert(DELTA || (JP & (JP - 1)) == 0, "draft bucket");
    static constexpr int JPP = JP <= 1 ? 1 : 2 << ilog2(JP - 1);  // JP rounded up to a power of two
    // bf16 row blocks of GDN heads (P = 128: both blocks of a head form one
    // M = 128 operand) are dotted on the tensor cores: D[P x 16] = S_c^T-view x
    // [the JP dot vectors, zero padded], in TMEM
    static constexpr bool UMMA = KIND == RS_GDN && P == 128 && N % 16 == 0 && JP <= 16;
    static constexpr int UMMA_N = 16;                     // MMA N (vectors, padded)
    static constexpr int UMMA_TCOLS = 32;                 // TMEM columns: two D buffers
    // the B operand: bf16 vectors as K-major 8 x 8 core matrices, one group of
    // 8 vectors (two when JP > 8); a unit uses it instead of the fp32 vectors
    static constexpr int QB_BYTES = (JP > 8 ? 2 : 1) * N * 16;
};

// Where a consumer warp's lanes sit in a stage of element type TE.  A row of
// the slab is NCB 128-byte lines; warp w owns CPW 16-byte chunks of line
// position cb = w / WPC; lane = cg + CPW * rg takes chunk cg in the rows
// row(rg) + RGW * k of every row block.  One shared-memory phase of 8 lanes
// reads CPW chunks in each of 8/CPW rows; row(rg) rotates the low bits of rg
// by SH = log2(CPW / NCB) (0 or 1) so that those rows differ in the line bits
// just above the chunk bits: the 8 chunks then fall in 8 different bank groups
// under the swizzle.
template <class C, typename TE>
struct WGeo {
    static constexpr int ESZ = sizeof(TE), VEC = 16 / ESZ;  // elements per 16-byte chunk
    static constexpr int NCB = C::P * ESZ / 128;            // lines per row = row blocks (stages) per slab
    static constexpr int WPC = C::NCW / NCB;                // warps per line position
    static constexpr int CPW = 8 / WPC;                     // chunks per warp
    static constexpr int LCG = ilog2(CPW);
    static constexpr int RGW = 32 / CPW;                    // row groups per warp
    static constexpr int LR = ilog2(RGW);
    static constexpr int LPH = ilog2(8 / CPW);              // log2 rows per shared-memory phase
    static constexpr int SH = ilog2(CPW / NCB);              // row rotation
    static constexpr int RB = C::N / NCB;                   // rows per row block
    static constexpr int RK = RB / RGW;                     // rows per lane per row block
    static constexpr int LSTRIDE = RGW * NCB;               // lines between a lane's rows
    static constexpr int CBE = 128 / ESZ;                   // elements per line
    static constexpr int JN = C::template jn<VEC>();        // dot vectors per pass
    static constexpr int NPASS = C::JP / JN;                // passes over the staged head
    static constexpr int M = VEC * JN;                      // partial sums per lane and pass
    static_assert(NCB >= 1 && C::NCW % NCB == 0 && CPW * WPC == 8 && CPW * C::NCW == 8 * NCB, "warp tiling");
    static_assert(SH <= 1 && LSTRIDE % 8 == 0 && RGW >= (1 << (LPH + SH)), "a lane keeps one swizzle phase");
    static_assert(RB * NCB * 128 == C::STAGE && RB % RGW == 0, "a row block is one stage");
    // the row (within a row block) of row group rg
    static __device__ __forceinline__ int row_of(int rg) {
        if constexpr (SH == 0) {
            return rg;
        } else {
            constexpr int MSK = (2 << LPH) - 1;
            const int low = rg & MSK;
            return (rg & ~MSK) | (((low << 1) | (low >> LPH)) & MSK);
        }
    }
};

// Header of a unit context: the plan and the unit's place.
struct UnitHdr {
    SeqPlan s;
    int b, h0;
};

// Shared-memory carve-up of one pipeline, byte offsets from a 1024-byte
// aligned base (stages first, so every stage is 1024-byte aligned as the
// swizzle requires).  The unit context (ctx*, offsets within one context) is
// double-buffered; the prep warps' scratch (d1, d2, sr, cst) and the consumer
// warps' scratch (fcf, unew) are not.  Value records (Mamba-2 x, GDN u) are
// read from global memory where needed: a fold gathers them into fcf (fw_r v_r
// for the warp's P/NCW columns, fold_chunk(cap) records at a time); unew holds
// the u of the launch's own records, written and read by the same warp.
struct RSmem {
    int stages, bars, plans, abort, tmem, d1, d2, sr, cst, fcf, unew, ctx0, ctx_bytes;
    int hdr, kraw, ar, vb, bt, c1, c2, g1, g2, fw, gF, pre1, qs, gv, fk;  // within a context
    int total;
};

__host__ __device__ inline int al16(int x) { return (x + 15) & ~15; }

// Units the planner lane may plan ahead of the prep warps.
constexpr int kPlanRing = 4;
// Records whose fold coefficients a consumer warp gathers at a time: 16 (a
// fold takes at most L = 16 records, so one gather per folded head) up to a
// 24-record buffer, else 8.
__host__ __device__ inline int fold_chunk(int cap) { return cap <= 24 ? 16 : 8; }

template <class C>
__host__ __device__ inline RSmem replay_smem(int cap, int HU, int NS) {
    constexpr int TMAX = C::TMAX, P = C::P, N = C::N;
    constexpr bool GDN = C::DELTA, KDA = C::KDA;  // (GDN: either delta-rule family)
    RSmem s;
    int o = 0;
    s.stages = o; o += NS * C::STAGE;
    s.bars = o;   o += al16((2 * NS + 6 + 2 * kPlanRing + 4) * 8);  // stage, context, plan, MMA barriers
    s.plans = o;  o += al16(kPlanRing * (int)sizeof(UnitHdr));
    s.abort = o;  o += 16;
    s.tmem = o;   o += 16;                                          // TMEM address of the D buffers
    s.d1 = o;     o += KDA ? 0 : al16(cap * TMAX * 4);              // k_r . q_i (GDN: k_r . k_{m_i})
    s.d2 = o;     o += GDN && !KDA ? al16(cap * TMAX * 4) : 0;      // GDN k_r . q_i
    s.sr = o;     o += al16(HU * cap * 4);                          // Mamba-2 dt_r
    s.cst = o;    o += al16(2 * HU * 4);                            // Mamba-2 A_h, D_h
    s.fcf = o;    o += al16(fold_chunk(cap) * P * 4);               // consumer warps' fold coefficients
    // GDN: u of this launch's records, written and read by the consumer warps
    // (each warp its own columns) within one unit: not double-buffered
    s.unew = o;   o += GDN ? al16(HU * TMAX * P * 4) : 0;
    int c = 0;
    s.hdr = c;    c += al16((int)sizeof(UnitHdr));
    s.kraw = c;   c += al16((cap + TMAX) * N * 2);                  // bf16 keys (rows < cap), queries (cap + i)
    s.ar = c;     c += KDA ? 0 : al16(HU * cap * 4);                // decays alpha_r (KDA: read in the scan)
    s.vb = c;     c += GDN ? al16(TMAX * HU * P * 2) : 0;           // GDN drafts' v (bf16)
    s.bt = c;     c += GDN ? al16(TMAX * HU * 4) : 0;               // GDN drafts' beta
    s.c1 = c;     c += al16(HU * TMAX * cap * 4);
    s.c2 = c;     c += GDN ? al16(HU * TMAX * cap * 4) : 0;
    s.g1 = c;     c += al16(HU * TMAX * 4);
    s.g2 = c;     c += al16(HU * TMAX * 4);
    s.fw = c;     c += al16(HU * cap * 4);
    s.gF = c;     c += al16(HU * 4);
    // Mamba-2: record parts of the outputs (GDN, KDA: summed by the consumer warps)
    s.pre1 = c;   c += GDN ? 0 : al16(HU * TMAX * P * 4);
    // fp32 dot vectors [QC][N][QW] (KDA: one set per head), or (tensor-core
    // units) the bf16 B operand
    s.qs = c;     c += al16(KDA ? HU * N * C::JP * 4 : (C::UMMA && C::QB_BYTES > N * C::JP * 4 ? C::QB_BYTES : N * C::JP * 4));
    // KDA fold: gamma(F-1) per key channel [HU][N], the decayed keys
    // w_r(F-1) (.) k_r of the folded records [HU][cap][N], fp32
    s.gv = c;     c += KDA ? al16(HU * N * 4) : 0;
    s.fk = c;     c += KDA ? al16(HU * cap * N * 4) : 0;
    s.ctx_bytes = c;
    s.ctx0 = o;   o += 2 * c;
    s.total = o;
    return s;
}

// Whether a launch dots its bf16 blocks on the tensor cores: two-precision
// checkpoints (bf16 reads never fold, so nothing but the MMAs reads a bf16
// stage).  The ring depth is then even, so that the two blocks of a head (ring
// positions q0, q0 + 1 with q0 even) are adjacent stages, and the bf16 copy is
// streamed in column blocks: a stage holds one 64-column half of the slab for
// all N keys, line n = key n, the layout of an MN-major operand.
template <class C>
__host__ __device__ inline bool umma_prec(const ReplayParams &p) {
    return C::UMMA && p.prec == RS_PREC_TWO && p.ckpt_lp != nullptr;
}

// Shared memory of one pipeline: its carve-up, rounded to the 1024-byte
// alignment of the next pipeline's stages.
__host__ __device__ inline int pipe_bytes(const RSmem &L) { return (L.total + 1023) & ~1023; }

// Where a pipeline sits in its CTA.  A CTA runs one pipeline (NT threads), or
// two side by side (2 NT threads, two carve-ups): kernels that hold tensor
// memory are resident one CTA per SM, so they pair their pipelines in one CTA.
struct PipeCtx {
    int u0, ustride;        // the pipeline's units: u0, u0 + ustride, ...
    int tid;                // thread index within the pipeline
    int bar_prep;           // named barrier of the pipeline's prep warps
    bool tc;                // bf16 blocks are dotted on the tensor cores
    const uint32_t *tslot;  // TMEM address of the CTA's allocation
    uint32_t tcol;          // the pipeline's first TMEM column
};

// VEC consecutive bf16 values (VEC = 4: 8-byte aligned, VEC = 8: 16-byte aligned) as fp32.
template <int VEC>
__device__ __forceinline__ void load_bf16_vec(const uint16_t *src, float (&out)[VEC]) {
    if constexpr (VEC == 8) {
        unpack<uint16_t, 8>(ld_u4(src), out);
    } else {
        static_assert(VEC == 4, "4 or 8 values");
        const uint2 u = *reinterpret_cast<const uint2 *>(src);
        out[0] = bf2f(u.x & 0xffffu); out[1] = __uint_as_float(u.x & 0xffff0000u);
        out[2] = bf2f(u.y & 0xffffu); out[3] = __uint_as_float(u.y & 0xffff0000u);
    }
}

// VEC consecutive fp32 values (16-byte aligned).
template <int VEC>
__device__ __forceinline__ void load_f32_vec(const float *src, float (&out)[VEC]) {
#pragma unroll
    for (int c = 0; c < VEC / 4; ++c) {
        const float4 f = reinterpret_cast<const float4 *>(src)[c];
        out[4 * c] = f.x; out[4 * c + 1] = f.y; out[4 * c + 2] = f.z; out[4 * c + 3] = f.w;
    }
}

// Dot-vector slots J0 .. J0+JN-1 of key row n ([QC][N][QW] fp32 layout: the
// lanes of a warp read consecutive rows, i.e. consecutive addresses).
template <class C, int J0, int JN>
__device__ __forceinline__ void load_q(const float *qs, int n, float (&qv)[JN]) {
    constexpr int QW = C::QW, N = C::N;
    static_assert(J0 % QW == 0 && JN % QW == 0, "whole vectors");
#pragma unroll
    for (int c = 0; c < JN / QW; ++c) {
        const float *src = qs + ((size_t)(J0 / QW + c) * N + n) * QW;
        if constexpr (QW == 4) {
            const float4 f = *reinterpret_cast<const float4 *>(src);
            qv[4 * c] = f.x; qv[4 * c + 1] = f.y; qv[4 * c + 2] = f.z; qv[4 * c + 3] = f.w;
        } else if constexpr (QW == 2) {
            const float2 f = *reinterpret_cast<const float2 *>(src);
            qv[2 * c] = f.x; qv[2 * c + 1] = f.y;
        } else {
            qv[c] = *src;
        }
    }
}

// Sum of v over the RGW row-group lanes of a warp (lane bits LCG and up), by
// recursive halving while more than NV values remain per lane, then by
// butterfly.  Afterwards a lane holds, in v[0..NV), the totals of entries
// a0 .. a0+NV-1 with a0 = (rg >> (LR - H)) * NV, H = log2(M / NV) halvings.
template <int M, int SZ, int NV, int MASK, int LCG>
struct RowReduce {
    static __device__ __forceinline__ void run(float (&v)[M], int rg) {
        if constexpr (MASK >= 1) {
            if constexpr (SZ > NV) {
                constexpr int HALF = SZ / 2;
                const bool up = (rg & MASK) != 0;
#pragma unroll
                for (int i = 0; i < HALF; ++i) {
                    const float send = up ? v[i] : v[i + HALF];
                    const float keep = up ? v[i + HALF] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, MASK << LCG);
                }
                RowReduce<M, HALF, NV, MASK / 2, LCG>::run(v, rg);
            } else {
#pragma unroll
                for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], MASK << LCG);
                RowReduce<M, SZ, NV, MASK / 2, LCG>::run(v, rg);
            }
        }
    }
};

// The lane's VEC columns times dot-vector slots J0 .. J0+JN-1 over the lane's
// RK rows of one staged row block (rows row0, row0 + RGW, ... of the slab),
// added to acc[e * JN + jj].
template <class C, typename TE, int J0>
__device__ __forceinline__ void dot_rows(const uint8_t *lane_base, const float *qs, int row0,
                                         float (&acc)[WGeo<C, TE>::M]) {
    using W = WGeo<C, TE>;
    constexpr int VEC = W::VEC, RGW = W::RGW, JN = W::JN;
#pragma unroll
    for (int k = 0; k < W::RK; ++k) {
        float sv[VEC], qv[JN];
        unpack<TE, VEC>(ld_u4(lane_base + (size_t)k * RGW * W::NCB * 128), sv);
        load_q<C, J0, JN>(qs, row0 + k * RGW, qv);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
#pragma unroll
            for (int jj = 0; jj < JN; ++jj) acc[e * JN + jj] = fmaf(sv[e], qv[jj], acc[e * JN + jj]);
    }
}

// Sums over the warp's row groups, keeping at least KEEP entries per lane.
template <class C, typename TE, int KEEP>
__device__ __forceinline__ void reduce_rows(float (&acc)[WGeo<C, TE>::M], int rg) {
    using W = WGeo<C, TE>;
    constexpr int NV = W::M / W::RGW > KEEP ? W::M / W::RGW : KEEP;
    RowReduce<W::M, W::M, NV, W::RGW / 2, W::LCG>::run(acc, rg);
}

// ---------------------------------------------------------------------------
// Planner (one lane of the producer warp): reads each unit's pointers, takes
// part in the pointer update, and hands the plan to the prep warps through a
// ring of kPlanRing slots, so that the pointer reads and the arrival atomic of
// later units overlap the prep warps' work on the current one.  A plan with
// b = -1 ends the pipeline.  Units are assigned round-robin (u0, u0 + ustride,
// ...): handing them out from one counter, as the row-split pipeline does,
// measured slower here (the two-precision GDN round 0.369 against 0.324 ms,
// same GPU).
template <class C>
__device__ __forceinline__ void planner(const ReplayParams &p, uint8_t *sm, const RSmem &L, int units, int HU,
                                        int NS, const PipeCtx &pc) {
    uint64_t *pfull = reinterpret_cast<uint64_t *>(sm + L.bars) + 2 * NS + 6, *pempty = pfull + kPlanRing;
    UnitHdr *plans = reinterpret_cast<UnitHdr *>(sm + L.plans);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.abort);
    const unsigned upseq = p.H / HU;
    for (int cu = 0, u = pc.u0;; ++cu, u += pc.ustride) {
        const int slot = cu % kPlanRing;
        if (!wait_or_abort(pempty + slot, ((cu / kPlanRing) & 1) ^ 1, abort_flag, p.status)) return;
        if (u >= units) {
            plans[slot].b = -1;
            mbar_arrive(pfull + slot);
            return;
        }
        const int b = u / upseq;
        const SeqPlan s = plan_sequence(p, b);
        arrive_and_update(p, s, b, upseq, (u % upseq) == 0);
        plans[slot].s = s;
        plans[slot].b = b;
        plans[slot].h0 = (u % upseq) * HU;
        mbar_arrive(pfull + slot);  // release: the plan is visible to the prep warps
    }
}

// ---------------------------------------------------------------------------
// Producer: stream each unit's row blocks once the prep warps have planned it.
template <class C>
__device__ __forceinline__ void producer(const ReplayParams &p, uint8_t *sm, const RSmem &L, int units, int HU,
                                         int NS, const CUtensorMap *map_hp, const CUtensorMap *map_lp,
                                         const PipeCtx &pc) {
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.bars), *empty = full + NS, *cplan = empty + NS;
    uint64_t *cempty = cplan + 4;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.abort);
    int st = 0, ph = 0, issued = 0, cu = 0;
    bool stop = false;
    for (; !stop; ++cu) {
        const int buf = cu & 1;
        if (!wait_or_abort(cplan + buf, (cu >> 1) & 1, abort_flag, p.status)) break;
        const UnitHdr hd = *reinterpret_cast<const UnitHdr *>(sm + L.ctx0 + buf * L.ctx_bytes + L.hdr);
        if (hd.b < 0) break;  // the pipeline's last unit is streamed
        // the prep warps rebuild this context only after this arrival (and the
        // consumer warps'), so no plan phase can pass unread
        mbar_arrive(cempty + buf);
        if (!hd.s.work) continue;
        const bool lp = plan_reads_lp(p, hd.s);
        const bool colb = lp && pc.tc;  // bf16 column blocks for the tensor cores
        const CUtensorMap *map = lp ? map_lp : map_hp;
        const int ncb = C::P * (lp ? 2 : 4) / 128, rb_rows = C::N / ncb;
        for (int j = 0; j < HU && !stop; ++j) {
            for (int rb = 0; rb < ncb; ++rb) {
                if (!wait_or_abort(empty + st, ph ^ 1, abort_flag, p.status)) { stop = true; break; }
                mbar_arrive_expect_tx(full + st, C::STAGE);
                tma_load_4d(sm + L.stages + (size_t)st * C::STAGE, map, 0, colb ? rb : 0, colb ? 0 : rb * rb_rows,
                            hd.b * p.H + hd.h0 + j, full + st);
                ++issued;
                if (++st == NS) { st = 0; ph ^= 1; }
            }
        }
    }
    if (*abort_flag) {
        // drain: wait (bounded) for the copies this thread may still have in flight,
        // the last min(NS, issued) ones, walking the ring backwards
        int s = st, q = ph;
        for (int k = 0; k < NS && k < issued; ++k) {
            if (--s < 0) { s = NS - 1; q ^= 1; }
            mbar_wait(full + s, q);
        }
    }
}

// ---------------------------------------------------------------------------
// Where the fold of one head finds the value vector of record r: the
// committed records (r < hc) in the record buffer, this launch's records in
// the step inputs (Mamba-2 x) or in the context (GDN u).
struct FoldSrc {
    const uint8_t *committed;  // record buffer, slot 0 of this (sequence, head)
    const uint8_t *fresh;      // record hc of this (sequence, head)
    size_t slot_stride, fresh_stride;  // bytes between slots / between this launch's records
    int base, hc, cap;
    int u16;                   // GDN: the committed records keep u in bf16 (this launch's are fp32)
};

// Gathers fw_r v_r[p] for records r0 .. r0+nr-1 and the warp's WC = P/NCW
// value columns (from column wcol0 on) into the warp's scratch
// cfs[r - r0][WC], fp32.  The loads of a chunk are independent.
template <class C>
__device__ __forceinline__ void gather_fold_coefs(float *cfs, const FoldSrc &fs, const float *fw, int r0, int nr,
                                                  int j, int wcol0, int lane) {
    constexpr int WC = C::P / C::NCW, Q = WC / 4;  // four columns per item
    constexpr int VSZ = C::KIND == RS_MAMBA2 ? 2 : 4;
    __syncwarp();  // the previous chunk's coefficients have been read
    for (int i = lane; i < nr * Q; i += 32) {
        const int r = r0 + i / Q, c4 = i % Q;
        int sl = fs.base + r;
        if (sl >= fs.cap) sl -= fs.cap;
        // Mamba-2 x is bf16 throughout; GDN u is fp32, or bf16 in the buffer with RS_U_BF16
        const bool b16 = C::KIND == RS_MAMBA2 || (fs.u16 && r < fs.hc);
        const uint8_t *src = (r < fs.hc ? fs.committed + (size_t)sl * fs.slot_stride
                                        : fs.fresh + (size_t)(r - fs.hc) * fs.fresh_stride) +
                             (size_t)(wcol0 + 4 * c4) * (b16 ? 2 : VSZ);
        float v[4];
        if (b16) load_bf16_vec<4>(reinterpret_cast<const uint16_t *>(src), v);
        else load_f32_vec<4>(reinterpret_cast<const float *>(src), v);
        const float w = fw ? fw[j * fs.cap + r] : 1.f;
        *reinterpret_cast<float4 *>(cfs + (r - r0) * WC + 4 * c4) =
            make_float4(w * v[0], w * v[1], w * v[2], w * v[3]);
    }
    __syncwarp();
}

// As gather_fold_coefs for GDN and KDA records, without the factor fw_r
// (the caller applies it as it reads): the committed records' u go straight
// from global memory to the scratch with cp.async, all of a lane's copies in
// flight at once and no registers held; this launch's records (in shared
// memory) are copied directly.  bf16 u (RS_U_BF16) lands in the upper half of
// the item's 16-byte fp32 slot and is widened in place after the wait: each
// lane widens only the items it copied.
template <class C>
__device__ __forceinline__ void gather_fold_values_async(float *cfs, const FoldSrc &fs, int nr, int wcol0,
                                                         int lane) {
    static_assert(C::KIND != RS_MAMBA2, "GDN and KDA record values");
    constexpr int WC = C::P / C::NCW, Q = WC / 4;
    __syncwarp();  // the previous coefficients have been read
    const int esz = fs.u16 ? 2 : 4;
    for (int i = lane; i < nr * Q; i += 32) {
        const int r = i / Q, c4 = i % Q;
        float *dst = cfs + r * WC + 4 * c4;
        if (r < fs.hc) {
            int sl = fs.base + r;
            if (sl >= fs.cap) sl -= fs.cap;
            const uint8_t *src = fs.committed + (size_t)sl * fs.slot_stride + (size_t)(wcol0 + 4 * c4) * esz;
            if (fs.u16) cp_async8(dst + 2, src);
            else cp_async16(dst, src);
        } else {
            *reinterpret_cast<float4 *>(dst) = *reinterpret_cast<const float4 *>(
                fs.fresh + (size_t)(r - fs.hc) * fs.fresh_stride + (size_t)(wcol0 + 4 * c4) * 4);
        }
    }
    cp_async_wait_all();
    if (fs.u16) {
        for (int i = lane; i < min(nr, fs.hc) * Q; i += 32) {
            float *dst = cfs + (i / Q) * WC + 4 * (i % Q);
            float v[4];
            load_bf16_vec<4>(reinterpret_cast<const uint16_t *>(dst + 2), v);
            *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
    __syncwarp();
}

// The fold's factor of key row n: gF for one decay per head; gamma(F-1)[n]
// (gvh, the head's per-channel products) for KDA.
template <class C>
__device__ __forceinline__ float fold_row_scale(const float *gvh, float gf, int n) {
    if constexpr (C::KDA) return gvh[n];
    else return gf;
}

// Adds records r0 .. r0+nr-1 of the fold S_new = gF S_c + sum_r (fw_r v_r) k_r^T
// to the lane's RK rows (row0, row0 + RGW, ...) of one row block: o[k][e].
// KDA: the keys are the head's fp32 decayed keys fkh [cap][N] (w_r (.) k_r).
template <class C, typename TE>
__device__ __forceinline__ void fold_records(float (&o)[WGeo<C, TE>::RK][WGeo<C, TE>::VEC], const uint16_t *kraw,
                                             const float *fkh, const float *cfs, int lcol, int r0, int nr,
                                             int row0) {
    using W = WGeo<C, TE>;
    constexpr int VEC = W::VEC, RK = W::RK, RGW = W::RGW, N = C::N, WC = C::P / C::NCW;
    for (int r = 0; r < nr; ++r) {
        float cf[VEC];
        load_f32_vec<VEC>(cfs + r * WC + lcol, cf);
        const uint16_t *kr = kraw + (size_t)(r0 + r) * N + row0;
        const float *fr = C::KDA ? fkh + (size_t)(r0 + r) * N + row0 : nullptr;
#pragma unroll
        for (int k = 0; k < RK; ++k) {
            const float kv = C::KDA ? fr[k * RGW] : bf2f(kr[k * RGW]);
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[k][e] = fmaf(cf[e], kv, o[k][e]);
        }
    }
}

// Writes the folded rows of one row block: the checkpoint (both copies as
// present) or the materialise output.
template <class C, typename TE>
__device__ __forceinline__ void fold_store(const ReplayParams &p, const float (&o)[WGeo<C, TE>::RK][WGeo<C, TE>::VEC],
                                           int row0, int col0, size_t goff, bool materialize) {
    using W = WGeo<C, TE>;
    constexpr int VEC = W::VEC, RK = W::RK, RGW = W::RGW, P = C::P;
#pragma unroll
    for (int k = 0; k < RK; ++k) {
        const size_t off = goff + (size_t)(row0 + k * RGW) * P + col0;
        if (materialize) {
            store_f32<VEC>(p.out + off, o[k]);
        } else {
            if (p.ckpt_hp) store_f32<VEC>(p.ckpt_hp + off, o[k]);
            if (p.ckpt_lp) store_bf16<VEC>(p.ckpt_lp + off, o[k]);
        }
    }
}

// A position q of the stage ring as its stage (q mod NS) and the parity of
// its fill (q div NS, mod 2), advanced incrementally (no division by the
// run-time ring depth).  Every consumer warp waits for every stage in ring
// order and arrives once on each, after its last read; the producer refills a
// stage only when all have.  A parity wait cannot tell a phase from the one two
// phases later, so no warp may skip a stage or fall a ring behind.
struct Ring {
    int s;
    unsigned ph;
};
__device__ __forceinline__ Ring ring_add(Ring r, int n, int NS) {
    r.s += n;
    while (r.s >= NS) {
        r.s -= NS;
        r.ph ^= 1u;
    }
    return r;
}
__device__ __forceinline__ bool wait_stage(uint64_t *full, Ring q, volatile int *abort_flag, uint32_t *status,
                                           bool ok) {
    ok = ok && wait_or_abort(full + q.s, q.ph, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void release_stage(uint64_t *empty, Ring q) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty + q.s);
}

// Fold of the lane's columns of a head whose NCB row blocks are all staged
// (KDA: gvh and fkh are the head's per-channel products and decayed keys).
// Coefficients are gathered fc records at a time.  fp32 blocks keep the
// partial sums in place between chunks (each lane rewrites only its own
// elements), so each chunk is gathered once per head; bf16 blocks (shared-bf16
// checkpoints) keep them in registers, one row block at a time.  Each row
// block (ring position q0 + rb) is handed back as soon as its last read is
// done, so the next copies overlap the rest of the fold.
template <class C, typename TE>
__device__ __forceinline__ void fold_head(const ReplayParams &p, uint8_t *stages, int lane_off, Ring q0, int NS,
                                          uint64_t *empty, const uint16_t *kraw,
                                          float *cfs, const FoldSrc &fs, const float *fw, float gf, const float *gvh,
                                          const float *fkh, int F, int j, int row0, int col0, int wcol0, int lcol,
                                          size_t goff, bool materialize, int lane, int fc) {
    using W = WGeo<C, TE>;
    constexpr int VEC = W::VEC, RK = W::RK, RGW = W::RGW, NCB = W::NCB, RB = W::RB;
    constexpr size_t RSTEP = (size_t)RGW * NCB * 128;
    const int nch = F > 0 ? (F + fc - 1) / fc : 1;
    auto blk = [&](int rb) { return stages + (size_t)ring_add(q0, rb, NS).s * C::STAGE + lane_off; };
    if constexpr (sizeof(TE) == 4 && W::CPW == 8 && W::RK == 8) {
        if (nch == 1) {
            // One gather; for the fold the lane takes 8 consecutive rows
            // 8 rg .. 8 rg + 7 of each row block (instead of rows rg + RGW k),
            // so that a record's keys for them are one 16-byte load.  The 8
            // lanes of a shared-memory phase still read one whole line; the
            // line's swizzle phase alternates with the row (NCB lines per row).
            const int cg = lane & 7, rg = lane >> 3, cb = wcol0 / W::CBE;
            gather_fold_values_async<C>(cfs, fs, F > 0 ? F : 0, wcol0, lane);
            for (int rb = 0; rb < NCB; ++rb) {
                const uint8_t *sb = stages + (size_t)ring_add(q0, rb, NS).s * C::STAGE;
                float o[8][4];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int line = (8 * rg + k) * NCB + cb;
                    unpack<float, 4>(ld_u4(sb + line * 128 + ((cg ^ (line & 7)) << 4)), o[k]);
                    const float sc = fold_row_scale<C>(gvh, gf, rb * RB + 8 * rg + k);
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[k][e] *= sc;
                }
                release_stage(empty, ring_add(q0, rb, NS));  // the block is in registers
                const uint16_t *kr = kraw + rb * RB + 8 * rg;
                for (int r = 0; r < F; ++r) {
                    float cf[4], kv[8];
                    load_f32_vec<4>(cfs + r * (C::P / C::NCW) + lcol, cf);
                    const float w = fw[j * fs.cap + r];
#pragma unroll
                    for (int e = 0; e < 4; ++e) cf[e] *= w;
                    if constexpr (C::KDA) load_f32_vec<8>(fkh + (size_t)r * C::N + rb * RB + 8 * rg, kv);
                    else unpack<uint16_t, 8>(ld_u4(kr + (size_t)r * C::N), kv);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[k][e] = fmaf(cf[e], kv[k], o[k][e]);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const size_t off = goff + (size_t)(rb * RB + 8 * rg + k) * C::P + col0;
                    if (materialize) {
                        store_f32<4>(p.out + off, o[k]);
                    } else {
                        if (p.ckpt_hp) store_f32<4>(p.ckpt_hp + off, o[k]);
                        if (p.ckpt_lp) store_bf16<4>(p.ckpt_lp + off, o[k]);
                    }
                }
            }
            return;
        }
    }
    if constexpr (sizeof(TE) == 4) {
        for (int c = 0; c < nch; ++c) {
            const int r0 = c * fc, nr = F - r0 < fc ? F - r0 : fc;
            gather_fold_coefs<C>(cfs, fs, fw, r0, nr > 0 ? nr : 0, j, wcol0, lane);
            for (int rb = 0; rb < NCB; ++rb) {
                float o[RK][VEC];
#pragma unroll
                for (int k = 0; k < RK; ++k) {
                    unpack<TE, VEC>(ld_u4(blk(rb) + k * RSTEP), o[k]);
                    if (c == 0) {
                        const float sc = fold_row_scale<C>(gvh, gf, rb * RB + row0 + k * RGW);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) o[k][e] *= sc;
                    }
                }
                if (c == nch - 1) {
                    // the block is in registers; partial sums written into the
                    // stages by earlier chunks precede the copies this lets in
                    if (nch > 1) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    release_stage(empty, ring_add(q0, rb, NS));
                }
                fold_records<C, TE>(o, kraw, fkh, cfs, lcol, r0, nr > 0 ? nr : 0, rb * RB + row0);
                if (c == nch - 1) {
                    fold_store<C, TE>(p, o, rb * RB + row0, col0, goff, materialize);
                } else {
#pragma unroll
                    for (int k = 0; k < RK; ++k)
                        *reinterpret_cast<float4 *>(blk(rb) + k * RSTEP) = make_float4(o[k][0], o[k][1], o[k][2], o[k][3]);
                }
            }
        }
    } else {
        for (int rb = 0; rb < NCB; ++rb) {
            float o[RK][VEC];
#pragma unroll
            for (int k = 0; k < RK; ++k) {
                unpack<TE, VEC>(ld_u4(blk(rb) + k * RSTEP), o[k]);
                const float sc = fold_row_scale<C>(gvh, gf, rb * RB + row0 + k * RGW);
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[k][e] *= sc;
            }
            release_stage(empty, ring_add(q0, rb, NS));  // the block is in registers
            for (int c = 0; c < nch; ++c) {
                const int r0 = c * fc, nr = F - r0 < fc ? F - r0 : fc;
                gather_fold_coefs<C>(cfs, fs, fw, r0, nr > 0 ? nr : 0, j, wcol0, lane);
                fold_records<C, TE>(o, kraw, fkh, cfs, lcol, r0, nr > 0 ? nr : 0, rb * RB + row0);
            }
            fold_store<C, TE>(p, o, rb * RB + row0, col0, goff, materialize);
        }
    }
}

// One pass of a warp over a head's row blocks (ring positions q0 ..
// q0+NCB-1) for dot-vector slots J0 .. J0+JN-1.  A streamed head waits for,
// reads and hands back each block in turn; a held head's blocks are already
// resident and stay so.  Returns false on abort.
template <class C, typename TE, int J0>
__device__ __forceinline__ bool head_pass(float (&acc)[WGeo<C, TE>::M], const ReplayParams &p, const uint8_t *stages,
                                          int lane_off, Ring q0, int NS, uint64_t *full, uint64_t *empty,
                                          volatile int *abort_flag, const float *qs, int rg, bool hold) {
    using W = WGeo<C, TE>;
    bool ok = true;
#pragma unroll
    for (int a = 0; a < W::M; ++a) acc[a] = 0.f;
#pragma unroll 1
    for (int rb = 0; rb < W::NCB; ++rb) {
        const Ring q = ring_add(q0, rb, NS);
        if (!hold && !(ok = wait_stage(full, q, abort_flag, p.status, ok))) break;
        dot_rows<C, TE, J0>(stages + (size_t)q.s * C::STAGE + lane_off, qs, rb * W::RB + rg, acc);
        if (!hold) release_stage(empty, q);
    }
    return ok;
}

// ---------------------------------------------------------------------------
// KDA: the per-channel decay products of one unit, one warp per head and lane
// = key channels lane + 32 t.  With w_r(m) = prod_{s=r+1..m} alpha_s and
// gamma(m) = prod_{s<=m} alpha_s, both vectors over the key channels, the
// state after record m is S_m = S_c diag(gamma(m)) + sum_{r<=m} u_r
// (w_r(m) (.) k_r)^T, so for draft i at position m_i = hc + i:
//   S_{m_i - 1} diag(alpha_{m_i}) k_{m_i} = S_c (gamma(m_i) (.) k_{m_i})
//                                        + sum_{r<m_i} u_r ((w_r(m_i) (.) k_r) . k_{m_i})
//   y_i = S_{m_i} q_i = S_c (gamma(m_i) (.) q_i) + sum_{r<=m_i} u_r ((w_r(m_i) (.) k_r) . q_i)
// One reverse pass over the records keeps a running product per bound (the
// drafts' m_i and the fold's F-1) and writes
//   c1[i][r] = (w_r(m_i) (.) k_r) . k_{m_i} (r < m_i),  c2[i][r] = (w_r(m_i) (.) k_r) . q_i (r <= m_i),
//   the fold keys fk[r] = w_r(F-1) (.) k_r (r < F) and gv = gamma(F-1),
//   the head's dot vectors gamma(m_i) (.) k_{m_i} and gamma(m_i) (.) q_i,
// and the GDN factors it replaces as ones (g1 = g2 = fw = gF = 1), so that the
// consumers' recurrence u_i = beta_i (v_i - sk_i) and outputs follow unchanged.
template <class C>
__device__ __forceinline__ bool kda_scan(const ReplayParams &p, uint8_t *cx, const RSmem &L, const SeqPlan &s,
                                         const int b, const int h0, const int HU, const PipeCtx &pc) {
    constexpr int N = C::N, TMAX = C::TMAX, JP = C::JP, JPP = C::JPP, QW = C::QW;
    constexpr int NPL = N / 32, LJ = ilog2(JPP);
    static_assert(N % 32 == 0, "key channels per lane");
    const int tp = pc.tid - C::PREP0, lane = tp & 31, pw = tp >> 5;
    const int H = p.H, cap = p.cap;
    const int base = s.base, hc = s.hc, T = s.T;
    const int nrec = hc + T;
    // the fold's records: F - 1 is the last folded position
    const int F = (s.fold || p.mode == MODE_MATERIALIZE) ? s.F : 0;
    auto slot = [&](int r) {
        const int v = base + r;
        return v >= cap ? v - cap : v;
    };
    const uint16_t *kraw = reinterpret_cast<const uint16_t *>(cx + L.kraw);
    float *c1 = reinterpret_cast<float *>(cx + L.c1), *c2 = reinterpret_cast<float *>(cx + L.c2);
    float *g1 = reinterpret_cast<float *>(cx + L.g1), *g2 = reinterpret_cast<float *>(cx + L.g2);
    float *fw = reinterpret_cast<float *>(cx + L.fw), *gF = reinterpret_cast<float *>(cx + L.gF);
    float *qs = reinterpret_cast<float *>(cx + L.qs);
    float *gv = reinterpret_cast<float *>(cx + L.gv), *fk = reinterpret_cast<float *>(cx + L.fk);
    // Warps per head: with one head per unit (and up to three drafts, whose
    // exchange below fits the head's fold-key area) the three prep warps split
    // the records into contiguous chunks, the highest first; each first forms
    // its chunk's products per bound, takes the products of the chunks above
    // it from the others, then scans its chunk.  Otherwise one warp per head.
    constexpr bool SPLIT = TMAX <= 3;
    const int wph = (SPLIT && HU < C::NPW) ? C::NPW / HU : 1;
    const int per = (nrec + wph - 1) / wph;
    for (int task = pw; task < (wph > 1 ? HU * wph : HU); task += (wph > 1 ? HU * wph : C::NPW)) {
        const int hd = task % HU, ci = task / HU, hh = h0 + hd;
        const int hi = nrec - ci * per > 0 ? nrec - ci * per : 0, lo = hi - per > 0 ? hi - per : 0;
        float Pd[TMAX][NPL], PF[NPL];  // running products: prod_{s=r+1..m} alpha_s[n]
#pragma unroll
        for (int t = 0; t < NPL; ++t) {
            PF[t] = 1.f;
#pragma unroll
            for (int i = 0; i < TMAX; ++i) Pd[i][t] = 1.f;
        }
        auto alpha_src = [&](int r) {
            return r < hc ? p.buf_a + (((size_t)b * cap + slot(r)) * H + hh) * N
                          : p.alpha + (((size_t)b * T + (r - hc)) * H + hh) * N;
        };
        if (SPLIT && wph > 1) {
            // pass 1: this chunk's products per bound, exchanged through the
            // head's fold-key area [chunk][bound][N] (pass 2 writes it later)
            float Qd[SPLIT ? TMAX : 1][NPL], QF[NPL];
#pragma unroll
            for (int t = 0; t < NPL; ++t) {
                QF[t] = 1.f;
#pragma unroll
                for (int i = 0; i < TMAX; ++i) Qd[i][t] = 1.f;
            }
            for (int r = lo; r < hi; ++r) {
                const float *asrc = alpha_src(r);
#pragma unroll
                for (int t = 0; t < NPL; ++t) {
                    const float a = asrc[lane + 32 * t];
#pragma unroll
                    for (int i = 0; i < TMAX; ++i)
                        if (i < T && r <= hc + i) Qd[i][t] *= a;
                    if (r < F) QF[t] *= a;
                }
            }
            float *xq = fk + (size_t)hd * cap * N;
#pragma unroll
            for (int t = 0; t < NPL; ++t) {
#pragma unroll
                for (int i = 0; i < TMAX; ++i) xq[((size_t)ci * (TMAX + 1) + i) * N + lane + 32 * t] = Qd[i][t];
                xq[((size_t)ci * (TMAX + 1) + TMAX) * N + lane + 32 * t] = QF[t];
            }
            if (named_sync_or(pc.bar_prep, C::NPT, false)) return false;
            for (int c2i = 0; c2i < ci; ++c2i) {  // the chunks above this one
#pragma unroll
                for (int t = 0; t < NPL; ++t) {
#pragma unroll
                    for (int i = 0; i < TMAX; ++i) Pd[i][t] *= xq[((size_t)c2i * (TMAX + 1) + i) * N + lane + 32 * t];
                    PF[t] *= xq[((size_t)c2i * (TMAX + 1) + TMAX) * N + lane + 32 * t];
                }
            }
            if (named_sync_or(pc.bar_prep, C::NPT, false)) return false;  // read before pass 2 writes fk
        }
        // the drafts' keys and queries at the lane's channels, read once (up to
        // four drafts; more are read per record)
        constexpr bool HOIST = TMAX <= 4;
        float kd[HOIST ? TMAX : 1][NPL], qd[HOIST ? TMAX : 1][NPL];
        if constexpr (HOIST) {
#pragma unroll
            for (int i = 0; i < TMAX; ++i)
#pragma unroll
                for (int t = 0; t < NPL; ++t) {
                    kd[i][t] = i < T ? bf2f(kraw[(size_t)(hc + i) * N + lane + 32 * t]) : 0.f;
                    qd[i][t] = i < T ? bf2f(kraw[(size_t)(cap + i) * N + lane + 32 * t]) : 0.f;
                }
        }
        // the records' decay vectors are loaded CA records at a time, ahead of
        // their use (they come from L2 or HBM; the scan is sequential)
        constexpr int CA = TMAX <= 3 ? 8 : 4;
        // one query (standard steps): the chunk's per-lane partial dots are kept
        // and reduced across the warp together after the chunk, one 16-value
        // reduction instead of one per record
        constexpr bool BATCH = TMAX == 1 && CA * JPP == 16;
        for (int rc = hi - 1; rc >= lo; rc -= CA) {
            float vb[BATCH ? CA * JPP : 1];
#pragma unroll
            for (int e = 0; e < (BATCH ? CA * JPP : 1); ++e) vb[e] = 0.f;
            float ac[CA][NPL];
#pragma unroll
            for (int q = 0; q < CA; ++q) {
                const int r = rc - q;
                if (r >= lo) {
                    const float *asrc = alpha_src(r);
#pragma unroll
                    for (int t = 0; t < NPL; ++t) ac[q][t] = asrc[lane + 32 * t];
                }
            }
#pragma unroll
        for (int q = 0; q < CA; ++q) {
            const int r = rc - q;
            if (r < lo) break;
            float a[NPL], kr[NPL];
#pragma unroll
            for (int t = 0; t < NPL; ++t) {
                a[t] = ac[q][t];
                kr[t] = bf2f(kraw[(size_t)r * N + lane + 32 * t]);
            }
            if (T > 0) {
                // slots i < TMAX: (w (.) k_r) . k_{m_i}; TMAX + i: (w (.) k_r) . q_i
                float v[JPP];
#pragma unroll
                for (int jj = 0; jj < JPP; ++jj) v[jj] = 0.f;
#pragma unroll
                for (int i = 0; i < TMAX; ++i) {
                    if (i < T && r <= hc + i) {
#pragma unroll
                        for (int t = 0; t < NPL; ++t) {
                            const int n = lane + 32 * t;
                            const float wk = Pd[i][t] * kr[t];
                            const float kv = HOIST ? kd[HOIST ? i : 0][t] : bf2f(kraw[(size_t)(hc + i) * N + n]);
                            const float qv = HOIST ? qd[HOIST ? i : 0][t] : bf2f(kraw[(size_t)(cap + i) * N + n]);
                            v[i] = fmaf(wk, kv, v[i]);
                            v[TMAX + i] = fmaf(wk, qv, v[TMAX + i]);
                        }
                    }
                }
                if constexpr (BATCH) {
#pragma unroll
                    for (int jj = 0; jj < JPP; ++jj) vb[(BATCH ? q * JPP : 0) + jj] = v[jj];
                } else {
                    RowReduce<JPP, JPP, 1, 16, 0>::run(v, lane);
                    const int sh = 5 - LJ;
                    if ((lane & ((1 << sh) - 1)) == 0) {
                        const int jj = lane >> sh;
                        if (jj < TMAX) {
                            if (jj < T) c1[(hd * TMAX + jj) * cap + r] = r < hc + jj ? v[0] : 0.f;
                        } else if (jj < JP && jj - TMAX < T) {
                            const int i = jj - TMAX;
                            c2[(hd * TMAX + i) * cap + r] = r <= hc + i ? v[0] : 0.f;
                        }
                    }
                }
            }
            if (r < F) {
#pragma unroll
                for (int t = 0; t < NPL; ++t) fk[((size_t)hd * cap + r) * N + lane + 32 * t] = PF[t] * kr[t];
            }
#pragma unroll
            for (int t = 0; t < NPL; ++t) {
#pragma unroll
                for (int i = 0; i < TMAX; ++i)
                    if (i < T && r <= hc + i) Pd[i][t] *= a[t];
                if (r < F) PF[t] *= a[t];
            }
        }
            if constexpr (BATCH) {
                if (T > 0) {
                    // lane 2e holds entry e = q JPP + jj: record rc - q, slot jj
                    RowReduce<BATCH ? CA * JPP : 1, BATCH ? CA * JPP : 1, 1, 16, 0>::run(vb, lane);
                    const int e = lane >> 1, q = e / JPP, jj = e % JPP, r = rc - q;
                    if ((lane & 1) == 0 && r >= lo) {
                        if (jj < TMAX) {
                            if (jj < T) c1[(hd * TMAX + jj) * cap + r] = r < hc + jj ? vb[0] : 0.f;
                        } else if (jj < JP && jj - TMAX < T) {
                            const int i = jj - TMAX;
                            c2[(hd * TMAX + i) * cap + r] = r <= hc + i ? vb[0] : 0.f;
                        }
                    }
                }
            }
        }
        // the warp whose chunk ends at record 0 now holds gamma(m_i) and gamma(F - 1)
        if (lo != 0 || (hi == 0 && ci != 0)) continue;
        float *qh = qs + (size_t)hd * N * JP;
#pragma unroll
        for (int t = 0; t < NPL; ++t) {
            const int n = lane + 32 * t;
#pragma unroll
            for (int jj = 0; jj < JP; ++jj) {
                const int i = jj < TMAX ? jj : jj - TMAX;
                const int row = i < T ? (jj < TMAX ? hc + i : cap + i) : -1;
                qh[((size_t)(jj / QW) * N + n) * QW + jj % QW] =
                    row >= 0 ? Pd[i][t] * bf2f(kraw[(size_t)row * N + n]) : 0.f;
            }
            gv[(size_t)hd * N + n] = F > 0 ? PF[t] : 1.f;
        }
        if (lane < TMAX) g1[hd * TMAX + lane] = g2[hd * TMAX + lane] = 1.f;
        if (lane < F) fw[hd * cap + lane] = 1.f;
        if (lane == 0) gF[hd] = 1.f;
    }
    return true;
}

// ---------------------------------------------------------------------------
// Prep warps: build the context of one unit (everything but the slab stream)
// in the context buffer `cx`.  Returns false when the CTA aborts.
template <class C>
__device__ __forceinline__ bool prep_unit(const ReplayParams &p, uint8_t *sm, const RSmem &L, uint8_t *cx,
                                          const SeqPlan &s, const int b, const int h0, const int HU, const bool tcu,
                                          const PipeCtx &pc) {
    constexpr int KIND = C::KIND, P = C::P, N = C::N, TMAX = C::TMAX, NPT = C::NPT, JP = C::JP;
    const int tp = pc.tid - C::PREP0, lane = tp & 31, pw = tp >> 5;
    const int H = p.H, G = p.G, cap = p.cap;
    const int g = h0 / (H / G);
    const int base = s.base, hc = s.hc, T = s.T, F = s.F;
    const bool append = s.append;
    const int nrec = hc + T;
    // buffer slot of record r: base < cap and r < cap for every planned unit
    // (plan_sequence), so one conditional subtract replaces the division
    auto slot = [&](int r) {
        const int v = base + r;
        return v >= cap ? v - cap : v;
    };

    float *d1 = reinterpret_cast<float *>(sm + L.d1), *d2 = reinterpret_cast<float *>(sm + L.d2);
    float *sr = reinterpret_cast<float *>(sm + L.sr);
    float *cst = reinterpret_cast<float *>(sm + L.cst);      // A_h (HU), D_h (HU)
    uint16_t *kraw = reinterpret_cast<uint16_t *>(cx + L.kraw);
    float *ar = reinterpret_cast<float *>(cx + L.ar);
    uint16_t *vb = reinterpret_cast<uint16_t *>(cx + L.vb);
    float *bt = reinterpret_cast<float *>(cx + L.bt);
    float *c1 = reinterpret_cast<float *>(cx + L.c1), *c2 = reinterpret_cast<float *>(cx + L.c2);
    float *g1 = reinterpret_cast<float *>(cx + L.g1), *g2 = reinterpret_cast<float *>(cx + L.g2);
    float *fw = reinterpret_cast<float *>(cx + L.fw), *gF = reinterpret_cast<float *>(cx + L.gF);
    float *pre1 = reinterpret_cast<float *>(cx + L.pre1);
    float *qs = reinterpret_cast<float *>(cx + L.qs);

    // Mamba-2 step-5 tasks: one head, 8 value columns and a group of XDG drafts
    // (all drafts at once would leave most prep threads idle at two heads per
    // unit).  The first task's first 8 records' x are loaded now, so that their
    // latency overlaps the staging.
    constexpr int PC8 = P / 8;
    constexpr int XDG = TMAX >= 4 ? 2 : TMAX, XNG = TMAX / XDG;  // drafts per task, draft groups
    const int x_tasks = KIND == RS_MAMBA2 && T > 0 ? HU * PC8 * XNG : 0;
    const uint16_t *xbuf = static_cast<const uint16_t *>(p.buf_v);
    auto x_src = [&](int task, int r) {
        const int hd = (task / PC8) % HU, pc = task % PC8;
        return (r < hc ? xbuf + (((size_t)b * cap + slot(r)) * H + h0 + hd) * P
                       : p.x + (((size_t)b * T + (r - hc)) * H + h0 + hd) * P) + 8 * pc;
    };
    uint4 xv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) xv[t] = tp < x_tasks && t < nrec ? ld_u4(x_src(tp, t)) : make_uint4(0u, 0u, 0u, 0u);

    // GDN, KDA: the committed records' u (P fp32 per head and record) are read
    // by the consumer warps (the record parts of the outputs, and the fold's
    // coefficients) one unit later; bring their lines into L2 now
    if (C::DELTA && T > 0) {
        const int esz = p.u16 ? 2 : 4, lpu = P * esz / 128;  // 128-byte lines per record value
        for (int i2 = tp; i2 < HU * hc * lpu; i2 += NPT) {
            const int l = i2 % lpu, r = (i2 / lpu) % hc, hh = h0 + i2 / (lpu * hc);
            prefetch_l2(static_cast<const uint8_t *>(p.buf_v) + ((((size_t)b * cap + slot(r)) * H + hh) * P) * esz + l * 128);
        }
    }
    // KDA: the records' decay vectors (N fp32 per head and record) are read by
    // the sequential scan; bring their lines into L2 now, so that they arrive
    // while the staging below waits
    if (C::KDA) {
        constexpr int LPV = N * 4 / 128;  // 128-byte lines per decay vector
        for (int i2 = tp; i2 < HU * nrec * LPV; i2 += NPT) {
            const int l = i2 % LPV, r = (i2 / LPV) % nrec, hh = h0 + i2 / (LPV * nrec);
            const float *src = r < hc ? p.buf_a + (((size_t)b * cap + slot(r)) * H + hh) * N
                                      : p.alpha + (((size_t)b * T + (r - hc)) * H + hh) * N;
            prefetch_l2(src + l * 32);
        }
    }
    // ---- 1. one batch of cp.async copies for every small operand of the unit
    {
        constexpr int KC = N / 8;  // 16-byte chunks per key row
        for (int i2 = tp; i2 < (nrec + T) * KC; i2 += NPT) {
            const int rr = i2 / KC, c = i2 % KC;
            const uint16_t *src;
            if (rr < hc) src = p.buf_k + (((size_t)b * cap + slot(rr)) * G + g) * N;
            else if (rr < nrec) src = (KIND == RS_MAMBA2 ? p.Bm : p.k) + (((size_t)b * T + (rr - hc)) * G + g) * N;
            else src = (KIND == RS_MAMBA2 ? p.Cm : p.q) + (((size_t)b * T + (rr - nrec)) * G + g) * N;
            const int row = rr < nrec ? rr : cap + (rr - nrec);
            cp_async16(kraw + (size_t)row * N + 8 * c, src + 8 * c);
        }
        if (KIND == RS_MAMBA2) {
            // (the records' x are read straight from global memory where needed)
            // A (forms the new records' decays) and D (the skip term of the
            // outputs) only exist for launches that append records; flush and
            // materialise pass neither
            for (int i2 = tp; i2 < (T > 0 ? HU : 0); i2 += NPT) {
                cp_async4(cst + i2, p.A + h0 + i2);
                if (p.D) cp_async4(cst + HU + i2, p.D + h0 + i2);
                else cst[HU + i2] = 0.f;
            }
        } else {  // the drafts' v (bf16) and beta (the committed u are read where needed)
            constexpr int VC = P / 8;
            for (int i2 = tp; i2 < T * HU * VC; i2 += NPT) {
                const int c = i2 % VC, hd = (i2 / VC) % HU, i = i2 / (VC * HU);
                cp_async16(vb + ((size_t)i * HU + hd) * P + 8 * c, p.v + (((size_t)b * T + i) * H + h0 + hd) * P + 8 * c);
            }
            for (int i2 = tp; i2 < T * HU; i2 += NPT) {
                const int hd = i2 % HU, i = i2 / HU;
                cp_async4(bt + i2, p.beta + ((size_t)b * T + i) * H + h0 + hd);
            }
        }
        // decays and value scales (KDA: the decay vectors are read by the scan)
        for (int i2 = tp; i2 < (C::KDA ? 0 : HU * nrec); i2 += NPT) {
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
    if (named_sync_or(pc.bar_prep, NPT, false)) return false;

    // ---- 2. new records' decays; appends; the fp32 dot vectors
    if (C::KDA && append) {  // the drafts' decay vectors, [H][N] per record
        constexpr int NC4 = N / 4;
        for (int i2 = tp; i2 < T * HU * NC4; i2 += NPT) {
            const int c = i2 % NC4, hd = (i2 / NC4) % HU, i = i2 / (NC4 * HU), hh = h0 + hd;
            const float4 a = reinterpret_cast<const float4 *>(p.alpha + (((size_t)b * T + i) * H + hh) * N)[c];
            reinterpret_cast<float4 *>(p.buf_a + (((size_t)b * cap + slot(hc + i)) * H + hh) * N)[c] = a;
        }
    }
    for (int i2 = tp; i2 < (C::KDA ? 0 : HU * T); i2 += NPT) {
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
            for (int i2 = tp; i2 < T * (N / 8); i2 += NPT) {
                const int i = i2 / (N / 8), c = i2 % (N / 8);
                uint16_t *dst = p.buf_k + (((size_t)b * cap + slot(hc + i)) * G + g) * N;
                reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(kraw + (size_t)(hc + i) * N)[c];
            }
        }
        // (Mamba-2: the new records' x are appended by the step-5 tasks)
    }
    // the key row that holds dot-vector slot jj: Mamba-2 C_jj; GDN k_{hc+jj}
    // (jj < TMAX) or q_{jj-TMAX}; -1 for the slots past the launch's drafts
    auto slot_row = [&](int jj) {
        if (KIND == RS_MAMBA2) return jj < T ? cap + jj : -1;
        if (jj < TMAX) return jj < T ? hc + jj : -1;
        return jj - TMAX < T ? cap + jj - TMAX : -1;
    };
    if (C::UMMA && T > 0 && tcu) {
        // the tensor cores' B operand (bf16): slot jj's keys 8c .. 8c+7 form
        // row jj % 8 of core matrix (jj / 8, c), core matrices 128 bytes apart
        // along the keys and N*16 bytes apart across groups of 8 slots; slots
        // past the launch's vectors are zero
        constexpr int KC = N / 8, NB = C::QB_BYTES / (N * 2);
        uint8_t *qb = reinterpret_cast<uint8_t *>(qs);
        for (int i2 = tp; i2 < NB * KC; i2 += NPT) {
            const int jj = i2 / KC, c = i2 % KC;
            const int row = jj < JP ? slot_row(jj) : -1;
            const uint4 v = row >= 0 ? ld_u4(kraw + (size_t)row * N + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(qb + (jj / 8) * (KC * 128) + c * 128 + (jj % 8) * 16) = v;
        }
        fence_proxy_async_smem();  // read by the tensor cores (async proxy)
    } else if (T > 0 && !C::KDA) {  // (KDA: per head, after the scan)
        // one key row n per task: its JP slots as fp32, QW at a time
        for (int n = tp; n < N; n += NPT) {
#pragma unroll
            for (int c = 0; c < C::QC; ++c) {
                float v[C::QW];
#pragma unroll
                for (int w = 0; w < C::QW; ++w) {
                    const int row = slot_row(c * C::QW + w);
                    v[w] = row >= 0 ? bf2f(kraw[(size_t)row * N + n]) : 0.f;
                }
                float *dst = qs + ((size_t)c * N + n) * C::QW;
                if constexpr (C::QW == 4) *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                else if constexpr (C::QW == 2) *reinterpret_cast<float2 *>(dst) = make_float2(v[0], v[1]);
                else dst[0] = v[0];
            }
        }
    }

    // ---- 3. key . dot-vector products d(r, jj) = k_r . v_jj (Mamba-2: d1 = k_r . q_i;
    // GDN: d1 = k_r . k_{m_i}, d2 = k_r . q_i): one warp per record at a time,
    // lane = key rows lane + 32 t; the slot vectors are read once per warp
    // from the staged bf16 rows, then a recursive-halving warp reduction
    // leaves slot jj's sum in lanes jj << (5 - log2 JP)
    if (T > 0 && !C::KDA) {
        constexpr int JPP = C::JPP, NPL = N / 32, LJ = ilog2(JPP);  // padded to a power of two
        constexpr bool HOIST = NPL * JPP <= 32;
        float qv[HOIST ? NPL : 1][JPP];
        auto slot_vals = [&](int t, float (&v)[JPP]) {
#pragma unroll
            for (int jj = 0; jj < JPP; ++jj) {
                const int row = jj < JP ? slot_row(jj) : -1;
                v[jj] = row >= 0 ? bf2f(kraw[(size_t)row * N + lane + 32 * t]) : 0.f;
            }
        };
        if constexpr (HOIST) {
#pragma unroll
            for (int t = 0; t < NPL; ++t) slot_vals(t, qv[t]);
        }
        for (int r = pw; r < nrec; r += C::NPW) {
            float acc[JPP];
#pragma unroll
            for (int jj = 0; jj < JPP; ++jj) acc[jj] = 0.f;
#pragma unroll
            for (int t = 0; t < NPL; ++t) {
                const float kv = bf2f(kraw[(size_t)r * N + lane + 32 * t]);
                if constexpr (!HOIST) slot_vals(t, qv[0]);
#pragma unroll
                for (int jj = 0; jj < JPP; ++jj) acc[jj] = fmaf(kv, qv[HOIST ? t : 0][jj], acc[jj]);
            }
            RowReduce<JPP, JPP, 1, 16, 0>::run(acc, lane);
            const int sh = 5 - LJ;
            if ((lane & ((1 << sh) - 1)) == 0) {
                const int jj = lane >> sh;
                if (KIND == RS_MAMBA2) {
                    if (jj < T) d1[r * TMAX + jj] = acc[0];
                } else if (jj < TMAX) {
                    if (jj < T) d1[r * TMAX + jj] = acc[0];
                } else if (jj - TMAX < T) {
                    d2[r * TMAX + jj - TMAX] = acc[0];
                }
            }
        }
    }
    if (named_sync_or(pc.bar_prep, NPT, false)) return false;

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
    if constexpr (C::KDA) {
        if (!kda_scan<C>(p, cx, L, s, b, h0, HU, pc)) return false;
    } else
    for (int hd = pw; hd < HU; hd += C::NPW) {
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
    if (named_sync_or(pc.bar_prep, NPT, false)) return false;

    // ---- 5. the parts of the outputs that come from the records, per value column
    if (KIND == RS_MAMBA2 && T > 0) {
        // rec_i[p] = sum_{r <= m_i} c1[i][r] x_r[p] + D x_{m_i}[p]: one task per
        // head, 8 columns and XDG drafts; the records' x come from global
        // memory, 8 records' loads in flight at a time (the first task's first
        // 8 were issued before the staging).  The tasks of the first draft
        // group also append the new x.
        for (int task = tp; task < x_tasks; task += NPT) {
            const int pc = task % PC8, hd = (task / PC8) % HU, ig = task / (PC8 * HU), i0 = ig * XDG;
            const float d = cst[HU + hd];
            float a[XDG][8];
#pragma unroll
            for (int i = 0; i < XDG; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) a[i][e] = 0.f;
            for (int r0 = 0; r0 < nrec; r0 += 8) {
                if (r0 > 0 || task != tp) {
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        xv[t] = r0 + t < nrec ? ld_u4(x_src(task, r0 + t)) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int r = r0 + t;
                    if (r >= nrec) break;
                    if (append && r >= hc && ig == 0)
                        *reinterpret_cast<uint4 *>(const_cast<uint16_t *>(xbuf) +
                                                   (((size_t)b * cap + slot(r)) * H + h0 + hd) * P + 8 * pc) = xv[t];
                    float xf[8];
                    unpack<uint16_t, 8>(xv[t], xf);
#pragma unroll
                    for (int k = 0; k < XDG; ++k) {
                        const int i = i0 + k;
                        if (i < T && r <= hc + i) {
                            const float c = c1[(hd * TMAX + i) * cap + r] + (r == hc + i ? d : 0.f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) a[k][e] = fmaf(c, xf[e], a[k][e]);
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < XDG; ++k) {
                if (i0 + k < T) {
                    float4 *dst = reinterpret_cast<float4 *>(pre1 + (hd * TMAX + i0 + k) * P + 8 * pc);
                    dst[0] = make_float4(a[k][0], a[k][1], a[k][2], a[k][3]);
                    dst[1] = make_float4(a[k][4], a[k][5], a[k][6], a[k][7]);
                }
            }
        }
        if (named_sync_or(pc.bar_prep, NPT, false)) return false;
    }
    // (GDN, KDA: the committed-record parts of S_{m_i-1} k_{m_i} and S_{m_i} q_i
    // are summed by the consumer warps, each for its own columns)
    return true;
}

// ---------------------------------------------------------------------------
// Consumer warps: the heads of one unit from its context `cx`, each warp on
// its own value columns.  `it` is the ring position of the unit's first
// stage.  Returns false when the CTA aborts.
template <class C, bool TC, typename TE>
__device__ __forceinline__ bool consume_heads(const ReplayParams &p, uint8_t *sm, const RSmem &L, const uint8_t *cx,
                                              const SeqPlan &s, const int b, const int h0, const int HU,
                                              const int NS, Ring &it, const PipeCtx &pc, int &mseq, bool &inflight) {
    constexpr int KIND = C::KIND, P = C::P, N = C::N, TMAX = C::TMAX, JP = C::JP;
    using W = WGeo<C, TE>;
    constexpr int VEC = W::VEC, RGW = W::RGW, LR = W::LR, M = W::M, NCB = W::NCB, JN = W::JN, NPASS = W::NPASS;
    static_assert(NPASS == 1 || NPASS == 2 || (NPASS == 4 && C::DELTA), "passes");
    const int lane = pc.tid & 31, warp = pc.tid >> 5;
    const int H = p.H, cap = p.cap, mode = p.mode;
    const int base = s.base, hc = s.hc, T = s.T, F = s.F;
    const bool append = s.append, materialize = mode == MODE_MATERIALIZE;
    const bool keep = s.fold || materialize;  // the staged head is read again by the fold
    // buffer slot of record r: base < cap and r < cap for every planned unit
    // (plan_sequence), so one conditional subtract replaces the division
    auto slot = [&](int r) {
        const int v = base + r;
        return v >= cap ? v - cap : v;
    };

    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.bars), *empty = full + NS;
    uint64_t *mdone = full + 2 * NS + 6 + 2 * kPlanRing, *dfree = mdone + 2;  // tensor-core D buffers
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.abort);
    const uint16_t *kraw = reinterpret_cast<const uint16_t *>(cx + L.kraw);
    float *unew = reinterpret_cast<float *>(sm + L.unew);  // GDN: u of new records
    const float *ar = reinterpret_cast<const float *>(cx + L.ar);
    const uint16_t *vb = reinterpret_cast<const uint16_t *>(cx + L.vb);
    const float *bt = reinterpret_cast<const float *>(cx + L.bt);
    const float *c1 = reinterpret_cast<const float *>(cx + L.c1), *c2 = reinterpret_cast<const float *>(cx + L.c2);
    const float *g1 = reinterpret_cast<const float *>(cx + L.g1), *g2 = reinterpret_cast<const float *>(cx + L.g2);
    const float *fw = reinterpret_cast<const float *>(cx + L.fw), *gF = reinterpret_cast<const float *>(cx + L.gF);
    const float *pre1 = reinterpret_cast<const float *>(cx + L.pre1);
    const float *qs = reinterpret_cast<const float *>(cx + L.qs);
    const float *gv = reinterpret_cast<const float *>(cx + L.gv), *fk = reinterpret_cast<const float *>(cx + L.fk);

    const int cb = warp / W::WPC;                                  // the warp's line position in a row
    const int cg = lane & (W::CPW - 1), rg = lane >> W::LCG;      // chunk among the warp's, row group
    const int ch = (warp % W::WPC) * W::CPW + cg;                  // 16-byte chunk within the line
    const int col0 = cb * W::CBE + ch * VEC;                       // first value column of the lane
    const int row0 = W::row_of(rg);                                // the lane's first row in a row block
    const int line0 = row0 * NCB + cb;
    // later rows of the lane are LSTRIDE (a multiple of 8) lines further on: same swizzle
    const int lane_off = line0 * 128 + ((ch ^ (line0 & 7)) << 4);
    // the warp's value columns are contiguous: P / NCW of them from wcol0
    const int wcol0 = cb * W::CBE + (warp % W::WPC) * W::CPW * VEC, lcol = col0 - wcol0;
    const int fc = fold_chunk(cap);
    float *cfs = reinterpret_cast<float *>(sm + L.fcf) + (size_t)warp * fc * (P / C::NCW);
    // A head stays resident (all its row blocks) when the slab is read again
    // after the reduction: by further passes, or by the fold (which for GDN
    // takes in the u this launch computes).  Otherwise each row block is
    // handed back as soon as every consumer warp has read it.
    const bool hold = NPASS > 1 || keep;
    const uint8_t *stages = sm + L.stages;
    bool ok = true;
    Ring q0 = it;  // the head's first row block
    for (int j = 0; j < HU && ok; ++j, q0 = ring_add(q0, NCB, NS)) {
        const int hh = h0 + j;
        const size_t goff = ((size_t)b * H + hh) * ((size_t)N * P);
        // KDA: the head's own dot vectors, per-channel products and decayed keys
        const float *qsh = C::KDA ? qs + (size_t)j * N * JP : qs;
        const float *gvh = C::KDA ? gv + (size_t)j * N : nullptr;
        const float *fkh = C::KDA ? fk + (size_t)j * cap * N : nullptr;
        FoldSrc fs;
        const int csz = (KIND == RS_MAMBA2 || p.u16) ? 2 : 4;  // bytes per buffered value
        fs.committed = static_cast<const uint8_t *>(p.buf_v) + ((size_t)b * cap * H + hh) * P * csz;
        fs.slot_stride = (size_t)H * P * csz;
        fs.u16 = KIND != RS_MAMBA2 && p.u16;
        if (KIND == RS_MAMBA2) {
            fs.fresh = reinterpret_cast<const uint8_t *>(p.x) + ((size_t)b * T * H + hh) * P * 2;
            fs.fresh_stride = (size_t)H * P * 2;
        } else {
            fs.fresh = reinterpret_cast<const uint8_t *>(unew + (size_t)j * TMAX * P);
            fs.fresh_stride = (size_t)P * 4;
        }
        fs.base = base; fs.hc = hc; fs.cap = cap;
        if (T == 0) {  // flush / materialise: fold only, the head's row blocks all resident
            for (int rb = 0; rb < NCB && ok; ++rb) ok = wait_stage(full, ring_add(q0, rb, NS), abort_flag, p.status, ok);
            if (!ok) break;
            fold_head<C, TE>(p, const_cast<uint8_t *>(stages), lane_off, q0, NS, empty, kraw, cfs, fs, fw, gF[j], gvh,
                             fkh, F, j, row0, col0, wcol0, lcol, goff, materialize, lane, fc);
            continue;
        }
        if (hold)
            for (int rb = 0; rb < NCB && ok; ++rb) ok = wait_stage(full, ring_add(q0, rb, NS), abort_flag, p.status, ok);
        if (!ok) break;
        float acc[M];
        if constexpr (KIND == RS_MAMBA2) {
            // y_i[p] = gamma(m_i) (S_c q_i)[p] + rec_i[p]
            constexpr int NV = M / RGW > 1 ? M / RGW : 1;
            constexpr int HV = ilog2(M / NV);
            const int a0 = (rg >> (LR - HV)) * NV;
            const bool lead = (rg & ((1 << (LR - HV)) - 1)) == 0;
            auto outputs = [&](int j0) {
#pragma unroll
                for (int t = 0; t < NV; ++t) {
                    const int a = a0 + t, e = a / JN, i = j0 + a % JN;
                    if (lead && i < T) {
                        const int pp = col0 + e;
                        p.y[(((size_t)b * T + i) * H + hh) * P + pp] =
                            fmaf(g1[j * TMAX + i], acc[t], pre1[(j * TMAX + i) * P + pp]);
                    }
                }
            };
            ok = head_pass<C, TE, 0>(acc, p, stages, lane_off, q0, NS, full, empty, abort_flag, qsh, row0, hold);
            if (!ok) break;
            reduce_rows<C, TE, 1>(acc, rg);
            outputs(0);
            if constexpr (NPASS == 2) {
                head_pass<C, TE, JN>(acc, p, stages, lane_off, q0, NS, full, empty, abort_flag, qsh, row0, hold);
                reduce_rows<C, TE, 1>(acc, rg);
                outputs(JN);
            }
        } else {
            // GDN: per value column, the recurrence over the drafts.  sums[jj]
            // holds (S_c v_jj)[pp] of the lane's column pp: slots i < TMAX the
            // keys k_{m_i}, slots TMAX + i the queries q_i.
            float sums[JP];
            int pp;
            bool lead;
            // The committed records' parts, per draft i: rs1[i] = sum_{r<hc}
            // c1[i][r] u_r[pp] (of S_{m_i-1} k_{m_i}) and rs2[i] = sum c2[i][r] u_r[pp]
            // (of S_{m_i} q_i), for the column the lane holds after the dots; the
            // first UPF records' u are loaded now, so that their latency overlaps
            // the dots (the tensor cores' or the lane's own).
            constexpr int UPF = 8;
            const int pl = (TC && C::UMMA && sizeof(TE) == 2) ? 32 * warp + lane : col0 + (rg >> (LR - ilog2(VEC)));
            const size_t uoff = ((size_t)b * cap * H + hh) * P + pl, ustride = (size_t)H * P;
            const bool u16 = p.u16 != 0;
            // A record's u is loaded as the aligned 32-bit word that holds it
            // (bf16: the lane's half of two columns) and widened only where it
            // is used, so that no instruction waits on the load before the dots.
            const int esz = u16 ? 2 : 4;
            const unsigned ush = u16 && !(pl & 1) ? 16u : 0u, umask = u16 ? 0xffff0000u : 0xffffffffu;
            auto u_at = [&](int r) {  // committed record r's u at the lane's column, raw
                const size_t i = (uoff + slot(r) * ustride) * esz;
                return *reinterpret_cast<const unsigned *>(static_cast<const uint8_t *>(p.buf_v) + (i & ~(size_t)3));
            };
            auto u_val = [&](unsigned raw) { return __uint_as_float((raw << ush) & umask); };
            unsigned upf[UPF];
#pragma unroll
            for (int t = 0; t < UPF; ++t) upf[t] = t < hc ? u_at(t) : 0u;
            if constexpr (TC && C::UMMA && sizeof(TE) == 2) {
                // Tensor cores: D[p][jj] = sum_n S_c[n][p] v_jj[n] for the head's
                // two row blocks (M = 128 value columns, K = N keys, A read from
                // the staged 128-byte-swizzled lines as an MN-major operand, B the
                // unit's bf16 vectors).  Warp 0 issues after the copies landed and
                // the D buffer's previous readers are done; every warp then reads
                // its 32 columns.  Double-buffered D: mseq counts the MMA heads.
                constexpr int NLD = JP <= 2 ? 2 : JP <= 4 ? 4 : JP <= 8 ? 8 : 16;
                const int db = mseq & 1;
                const unsigned use = (unsigned)mseq >> 1;
                const uint32_t tbase = *reinterpret_cast<const volatile uint32_t *>(pc.tslot) + pc.tcol;
                if (warp == 0) {
                    if (!hold)
                        for (int rb = 0; rb < NCB && ok; ++rb) ok = wait_stage(full, ring_add(q0, rb, NS), abort_flag, p.status, ok);
                    if (ok && use > 0)
                        ok = __all_sync(0xffffffffu, wait_or_abort(dfree + db, (use - 1) & 1u, abort_flag, p.status));
                    if (ok && lane == 0) {
                        tc_fence_after_sync();
                        const uint32_t a0 = smem_u32(stages + (size_t)q0.s * C::STAGE), b0 = smem_u32(qs);
                        constexpr uint32_t idesc = umma_idesc_bf16(128, C::UMMA_N, true, false);
#pragma unroll
                        for (int ks = 0; ks < N / 16; ++ks)
                            umma_bf16(tbase + db * C::UMMA_N, umma_smem_desc(a0 + ks * 2048, C::STAGE, 1024, 2),
                                      umma_smem_desc(b0 + ks * 256, 128, JP > 8 ? N * 16 : 0, 0), idesc, ks > 0);
                        umma_commit(mdone + db);
                    }
                    inflight = ok;
                    __syncwarp();
                }
                ok = ok && __all_sync(0xffffffffu, wait_or_abort(mdone + db, use & 1u, abort_flag, p.status));
                if (!ok) break;
                if (warp == 0) inflight = false;
                tc_fence_after_sync();
                float dv[NLD];
                tmem_ld<NLD>(tbase + ((uint32_t)(32 * warp) << 16) + db * C::UMMA_N, dv);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(dfree + db);  // this warp has read the D buffer
                if (!hold)  // the MMAs have read the row blocks
                    for (int rb = 0; rb < NCB; ++rb) release_stage(empty, ring_add(q0, rb, NS));
                ++mseq;
#pragma unroll
                for (int t = 0; t < JP; ++t) sums[t] = dv[t];
                pp = 32 * warp + lane;
                lead = true;
            } else {
                // CUDA cores: the reductions keep all sums of one column in one lane
                constexpr int HV = ilog2(VEC);
                const int e = rg >> (LR - HV);
                pp = col0 + e;
                lead = (rg & ((1 << (LR - HV)) - 1)) == 0;
                ok = head_pass<C, TE, 0>(acc, p, stages, lane_off, q0, NS, full, empty, abort_flag, qsh, row0, hold);
                if (!ok) break;
                reduce_rows<C, TE, JN>(acc, rg);
#pragma unroll
                for (int t = 0; t < JN; ++t) sums[t] = acc[t];
                if constexpr (NPASS >= 2) {
                    head_pass<C, TE, JN>(acc, p, stages, lane_off, q0, NS, full, empty, abort_flag, qsh, row0, hold);
                    reduce_rows<C, TE, JN>(acc, rg);
#pragma unroll
                    for (int t = 0; t < JN; ++t) sums[JN + t] = acc[t];
                }
                if constexpr (NPASS == 4) {
                    head_pass<C, TE, 2 * JN>(acc, p, stages, lane_off, q0, NS, full, empty, abort_flag, qsh, row0, hold);
                    reduce_rows<C, TE, JN>(acc, rg);
#pragma unroll
                    for (int t = 0; t < JN; ++t) sums[2 * JN + t] = acc[t];
                    head_pass<C, TE, 3 * JN>(acc, p, stages, lane_off, q0, NS, full, empty, abort_flag, qsh, row0, hold);
                    reduce_rows<C, TE, JN>(acc, rg);
#pragma unroll
                    for (int t = 0; t < JN; ++t) sums[3 * JN + t] = acc[t];
                }
            }
            float rs1[TMAX], rs2[TMAX];
#pragma unroll
            for (int i = 0; i < TMAX; ++i) rs1[i] = rs2[i] = 0.f;
            for (int r0 = 0; r0 < hc; r0 += UPF) {
                if (r0 > 0) {
#pragma unroll
                    for (int t = 0; t < UPF; ++t) upf[t] = r0 + t < hc ? u_at(r0 + t) : 0u;
                }
#pragma unroll
                for (int t = 0; t < UPF; ++t) {
                    const int r = r0 + t;
                    if (r < hc) {
                        const float uv = u_val(upf[t]);
#pragma unroll
                        for (int i = 0; i < TMAX; ++i) {
                            if (i < T) {
                                rs1[i] = fmaf(c1[(j * TMAX + i) * cap + r], uv, rs1[i]);
                                rs2[i] = fmaf(c2[(j * TMAX + i) * cap + r], uv, rs2[i]);
                            }
                        }
                    }
                }
            }
            float ud[TMAX];
#pragma unroll
            for (int i = 0; i < TMAX; ++i) {
                ud[i] = 0.f;
                if (i < T) {
                    const int m = hc + i;
                    float sk = g1[j * TMAX + i] * sums[i] + rs1[i];
                    const float *cc1 = c1 + (j * TMAX + i) * cap + hc;
#pragma unroll
                    for (int i3 = 0; i3 < TMAX; ++i3)
                        if (i3 < i) sk = fmaf(cc1[i3], ud[i3], sk);
                    // (KDA: alpha_{m} is inside the dot vectors and the coefficients)
                    const float am = C::KDA ? 1.f : ar[j * cap + m];
                    const float u = bt[i * HU + j] * (bf2f(vb[((size_t)i * HU + j) * P + pp]) - am * sk);
                    ud[i] = u;
                    float yv = g2[j * TMAX + i] * sums[TMAX + i] + rs2[i];
                    const float *cc2 = c2 + (j * TMAX + i) * cap + hc;
#pragma unroll
                    for (int i3 = 0; i3 < TMAX; ++i3)
                        if (i3 <= i) yv = fmaf(cc2[i3], ud[i3], yv);
                    if (lead) {
                        unew[((size_t)j * TMAX + i) * P + pp] = u;
                        if (append) {
                            const size_t ui = (((size_t)b * cap + slot(m)) * H + hh) * P + pp;
                            if (u16) static_cast<uint16_t *>(p.buf_v)[ui] = (uint16_t)f2bf(u);
                            else static_cast<float *>(p.buf_v)[ui] = u;
                        }
                        p.y[(((size_t)b * T + i) * H + hh) * P + pp] = yv;
                    }
                }
            }
            __syncwarp();  // the new records' u of the warp's columns are in the context
        }
        if (hold) {
            if (keep)
                fold_head<C, TE>(p, const_cast<uint8_t *>(stages), lane_off, q0, NS, empty, kraw, cfs, fs, fw, gF[j],
                                 gvh, fkh, F, j, row0, col0, wcol0, lcol, goff, materialize, lane, fc);
            else
                for (int rb = 0; rb < NCB; ++rb) release_stage(empty, ring_add(q0, rb, NS));
        }
    }
    it = q0;
    return ok;
}

// ---------------------------------------------------------------------------
// Role loops.
template <class C>
__device__ __forceinline__ void prep_loop(const ReplayParams &p, uint8_t *sm, const RSmem &L, int units, int HU,
                                          int NS, const PipeCtx &pc) {
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bars);
    uint64_t *cplan = bars + 2 * NS, *cfull = cplan + 2, *cempty = cfull + 2;
    uint64_t *pfull = cempty + 2, *pempty = pfull + kPlanRing;
    const UnitHdr *plans = reinterpret_cast<const UnitHdr *>(sm + L.plans);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.abort);
    const int tp = pc.tid - C::PREP0;
    for (int cu = 0;; ++cu) {
        const int buf = cu & 1;
        const bool ok = wait_or_abort(cempty + buf, ((cu >> 1) & 1) ^ 1, abort_flag, p.status);
        if (named_sync_or(pc.bar_prep, C::NPT, !ok)) return;  // the producer and every consumer warp are done with it
        uint8_t *cx = sm + L.ctx0 + buf * L.ctx_bytes;
        UnitHdr *hdr = reinterpret_cast<UnitHdr *>(cx + L.hdr);
        if (tp == 0) {
            // the unit's plan, from the planner lane
            const int slot = cu % kPlanRing;
            const bool got = wait_or_abort(pfull + slot, (cu / kPlanRing) & 1, abort_flag, p.status);
            if (got) {
                *hdr = plans[slot];
                mbar_arrive(pempty + slot);
                mbar_arrive(cplan + buf);  // release: the producer may stream the unit
            }
        }
        if (named_sync_or(pc.bar_prep, C::NPT, *abort_flag != 0)) return;
        const int b = hdr->b, h0 = hdr->h0;
        if (b < 0) {  // no more units: the consumer warps see the end plan too
            if (tp == 0) mbar_arrive(cfull + buf);
            return;
        }
        const SeqPlan s = hdr->s;
        if (s.work && !prep_unit<C>(p, sm, L, cx, s, b, h0, HU, pc.tc && plan_reads_lp(p, s), pc)) return;
        if (named_sync_or(pc.bar_prep, C::NPT, false)) return;  // the whole context is written
        if (tp == 0) mbar_arrive(cfull + buf);
    }
}

template <class C, bool TC>
__device__ __forceinline__ void consumer_loop(const ReplayParams &p, uint8_t *sm, const RSmem &L, int units, int HU,
                                              int NS, const PipeCtx &pc, int &mseq, bool &inflight) {
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bars);
    uint64_t *cfull = bars + 2 * NS + 2, *cempty = cfull + 2;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.abort);
    const int lane = pc.tid & 31;
    Ring it = {0, 0u};
    for (int cu = 0;; ++cu) {
        const int buf = cu & 1;
        const bool ok = __all_sync(0xffffffffu, wait_or_abort(cfull + buf, (cu >> 1) & 1, abort_flag, p.status));
        if (!ok) return;
        const uint8_t *cx = sm + L.ctx0 + buf * L.ctx_bytes;
        const UnitHdr hd = *reinterpret_cast<const UnitHdr *>(cx + L.hdr);
        if (hd.b < 0) return;
        if (hd.s.work) {
            const bool done = plan_reads_lp(p, hd.s)
                                  ? consume_heads<C, TC, uint16_t>(p, sm, L, cx, hd.s, hd.b, hd.h0, HU, NS, it, pc,
                                                                   mseq, inflight)
                                  : consume_heads<C, TC, float>(p, sm, L, cx, hd.s, hd.b, hd.h0, HU, NS, it, pc, mseq,
                                                                inflight);
            if (!done) return;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(cempty + buf);  // this warp is done with the context
    }
}

// TC: the kernel holds tensor memory (the bf16 blocks of two-precision
// launches are dotted on the tensor cores); such kernels are resident one CTA
// per SM, so they run PIPES = 2 pipelines side by side in one CTA.
template <class C, bool TC, int PIPES>
__global__ void __launch_bounds__(C::NT * PIPES, PIPES == 1 ? C::MIN_BLOCKS : 1)
    replay_pipe_kernel(const ReplayParams p, const __grid_constant__ CUtensorMap map_hp,
                       const __grid_constant__ CUtensorMap map_lp, int units, int HU, int NS) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the swizzle pattern is a function of the shared address: align the carve-up to 1024 bytes
    uint8_t *sm0 = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const RSmem L = replay_smem<C>(p.cap, HU, NS);
    const int pipe = PIPES == 1 ? 0 : (int)(threadIdx.x / C::NT);
    uint8_t *sm = sm0 + (size_t)pipe * pipe_bytes(L);
    PipeCtx pc;
    pc.u0 = blockIdx.x * PIPES + pipe;
    pc.ustride = gridDim.x * PIPES;
    pc.tid = threadIdx.x & (C::NT - 1);
    pc.bar_prep = 1 + pipe;  // named barriers 1 .. PIPES; PIPES + 1: every consumer warp of the CTA
    pc.tc = TC;
    pc.tslot = reinterpret_cast<const uint32_t *>(sm0 + L.tmem);
    pc.tcol = (uint32_t)(pipe * C::UMMA_TCOLS);
    if (pc.tid == 0) {
        uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bars);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bars + s, 1);             // full: the producer's expect_tx arrival
            mbar_init(bars + NS + s, C::NCW);   // empty: one arrival per consumer warp
        }
        uint64_t *pb = bars + 2 * NS;
        for (int k = 0; k < 2; ++k) {
            mbar_init(pb + k, 1);               // context planned: the prep warps (read by the producer)
            mbar_init(pb + 2 + k, 1);           // context full: the prep warps
            mbar_init(pb + 4 + k, C::NCW + 1);  // context empty: every consumer warp and the producer
        }
        for (int k = 0; k < kPlanRing; ++k) {
            mbar_init(pb + 6 + k, 1);               // plan full: the planner lane
            mbar_init(pb + 6 + kPlanRing + k, 1);   // plan empty: the prep warps
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(pb + 6 + 2 * kPlanRing + k, 1);       // MMA done: the issuing thread's commit
            mbar_init(pb + 8 + 2 * kPlanRing + k, C::NCW);  // D buffer read: every consumer warp
        }
        *reinterpret_cast<volatile int *>(sm + L.abort) = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const int warp = pc.tid >> 5;
    if constexpr (TC) {
        if (threadIdx.x < 32) tmem_alloc(reinterpret_cast<uint32_t *>(sm0 + L.tmem), C::UMMA_TCOLS * PIPES);
        tc_fence_before_sync();
    }
    __syncthreads();
    if constexpr (TC) tc_fence_after_sync();
    if (warp < C::NCW) {
        int mseq = 0;
        bool inflight = false;
        consumer_loop<C, TC>(p, sm, L, units, HU, NS, pc, mseq, inflight);
        if constexpr (TC) {
            // the TMEM goes back once no MMA is in flight and every consumer
            // warp of the CTA is done with it (also after an abort)
            if (warp == 0 && inflight) {
                uint64_t *mdone = reinterpret_cast<uint64_t *>(sm + L.bars) + 2 * NS + 6 + 2 * kPlanRing;
                mbar_wait(mdone + (mseq & 1), ((unsigned)mseq >> 1) & 1u);
            }
            tc_fence_before_sync();
            asm volatile("bar.sync %0, %1;" ::"n"(PIPES + 1), "n"(32 * C::NCW * PIPES) : "memory");
            if (threadIdx.x < 32) {
                tc_fence_after_sync();
                tmem_dealloc(*reinterpret_cast<const volatile uint32_t *>(pc.tslot), C::UMMA_TCOLS * PIPES);
            }
        }
    } else if (warp == C::NCW) {
        if (pc.tid == 32 * C::NCW) producer<C>(p, sm, L, units, HU, NS, &map_hp, &map_lp, pc);
        else if (pc.tid == 32 * C::NCW + 1) planner<C>(p, sm, L, units, HU, NS, pc);
    } else {
        prep_loop<C>(p, sm, L, units, HU, NS, pc);
    }
}

// ---------------------------------------------------------------------------
// Host side.

// Tensor map of a checkpoint copy viewed as [slabs][N][P/CB][CB] with CB
// elements = 128 bytes innermost; the box is one row block of one slab
// (CB x P/CB x N*CB/P x 1: contiguous in HBM, N x 128 bytes), landing in shared
// memory as 128-byte lines with the 128-byte swizzle.
bool encode_slab_map(CUtensorMap *map, const void *base, bool bf16, int P, int N, long long slabs, bool col_blocks);

// Launch shape: heads per unit, ring depth, CTAs per SM (pipelines per CTA
// for tensor-core kernels), shared memory.
struct LaunchShape {
    int HU, NS, per_sm, smem;
};

// Device limits used to size launches (queried once per device).
struct DeviceLimits {
    int sms, smem_per_sm, smem_per_block, reserved_per_block;
};
cudaError_t device_limits(DeviceLimits &d);

// CUDA-core kernels: two CTAs per SM (one CTA's per-unit phases overlap the
// other's stream), at least four stages each; else one CTA per SM with a
// deeper ring.
template <class C>
LaunchShape choose_shape(const ReplayParams &p, const DeviceLimits &dl) {
    const int hpg = p.H / p.G;
    static constexpr int kHU[] = {8, 4, 2, 1};
    LaunchShape best = {0, 0, 0, 0};
    for (int tier = C::MIN_BLOCKS == 2 ? 2 : 1; tier >= 1 && best.HU == 0; --tier) {
        const int budget = (tier == 2 ? dl.smem_per_sm / 2 - dl.reserved_per_block : dl.smem_per_block) - 1024;
        // a held head keeps all its row blocks resident: at least one fp32 slab of stages
        const int ns_max = tier == 2 ? 8 : 12, ns_min = C::P * 4 / 128 > 4 ? C::P * 4 / 128 : 4;
        for (int HU : kHU) {
            if (hpg % HU != 0) continue;
            const int other = replay_smem<C>(p.cap, HU, 0).total;
            int ns = (budget - other) / C::STAGE;
            if (ns > ns_max) ns = ns_max;
            if (ns < ns_min) continue;
            best = {HU, ns, tier, replay_smem<C>(p.cap, HU, ns).total + 1024};
            break;
        }
    }
    return best;
}

// Tensor-core kernels (one CTA per SM): two pipelines per CTA, each with half
// of the CTA's shared memory, at least four stages each; else one pipeline
// with a deeper ring.  The ring depth is even (a head's two bf16 blocks are
// adjacent stages).  per_sm holds the pipelines per CTA.
template <class C>
LaunchShape choose_shape_tc(const ReplayParams &p, const DeviceLimits &dl) {
    const int hpg = p.H / p.G;
    static constexpr int kHU[] = {8, 4, 2, 1};
    for (int pipes = 2; pipes >= 1; --pipes) {
        const int budget = pipes == 2 ? ((dl.smem_per_block - 1024) / 2) & ~1023 : dl.smem_per_block - 1024;
        const int ns_max = pipes == 2 ? 8 : 12, ns_min = C::P * 4 / 128 > 4 ? C::P * 4 / 128 : 4;
        for (int HU : kHU) {
            if (hpg % HU != 0) continue;
            const int other = replay_smem<C>(p.cap, HU, 0).total;
            int ns = (budget - other) / C::STAGE;
            if (ns > ns_max) ns = ns_max;
            ns &= ~1;
            if (ns < ns_min) continue;
            const RSmem L = replay_smem<C>(p.cap, HU, ns);
            return {HU, ns, pipes, (pipes == 2 ? 2 * pipe_bytes(L) : L.total) + 1024};
        }
    }
    return {0, 0, 0, 0};
}

template <class C, bool TC, int PIPES>
cudaError_t launch_kernel(const ReplayParams &p, const LaunchShape &sh, const DeviceLimits &dl,
                          cudaStream_t stream) {
    auto kern = replay_pipe_kernel<C, TC, PIPES>;
    static SmemGrants grants;  // this instantiation's opt-in, per device
    cudaError_t e = grant_smem(reinterpret_cast<const void *>(kern), dl.smem_per_block, grants);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::NT * PIPES, sh.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    CUtensorMap map_hp, map_lp;
    memset(&map_hp, 0, sizeof map_hp);
    memset(&map_lp, 0, sizeof map_lp);
    const long long slabs = (long long)p.B * p.H;
    if (p.ckpt_hp && !encode_slab_map(&map_hp, p.ckpt_hp, false, C::P, C::N, slabs, false))
        return cudaErrorInvalidValue;
    // the tensor cores read bf16 column blocks
    if (p.ckpt_lp && !encode_slab_map(&map_lp, p.ckpt_lp, true, C::P, C::N, slabs, TC))
        return cudaErrorInvalidValue;
    const int units = p.B * (p.H / sh.HU), ctas = (units + PIPES - 1) / PIPES;
    const int grid = ctas < dl.sms * per_sm ? ctas : dl.sms * per_sm;
    kern<<<grid, C::NT * PIPES, sh.smem, stream>>>(p, map_hp, map_lp, units, sh.HU, sh.NS);
    return cudaGetLastError();
}

template <class C>
cudaError_t launch_pipe(const ReplayParams &p, cudaStream_t stream) {
    DeviceLimits dl;
    cudaError_t e = device_limits(dl);
    if (e != cudaSuccess) return e;
    if constexpr (C::UMMA) {
        if (umma_prec<C>(p)) {
            const LaunchShape sh = choose_shape_tc<C>(p, dl);
            if (sh.HU != 0)
                return sh.per_sm == 2 ? launch_kernel<C, true, 2>(p, sh, dl, stream)
                                      : launch_kernel<C, true, 1>(p, sh, dl, stream);
        }
    }
    const LaunchShape sh = choose_shape<C>(p, dl);
    if (sh.HU == 0) return cudaErrorInvalidConfiguration;
    return launch_kernel<C, false, 1>(p, sh, dl, stream);
}

// Verify launches instantiate the draft-count buckets 1, 4 and 8 (GDN and KDA also 3).
template <int KIND, int P, int N>
cudaError_t dispatch_shape(const ReplayParams &p, cudaStream_t s) {
    const int T = p.mode == MODE_VERIFY ? p.T : 1;
    if (T <= 1) return launch_pipe<RCfg<KIND, P, N, 1>>(p, s);
    if (KIND != RS_MAMBA2 && T <= 3) return launch_pipe<RCfg<KIND, P, N, 3>>(p, s);
    if (T <= 4) return launch_pipe<RCfg<KIND, P, N, 4>>(p, s);
    return launch_pipe<RCfg<KIND, P, N, 8>>(p, s);
}

}  // namespace cols
}  // namespace rs
