// Per-sequence planning shared by the replay kernels: what one launch does to
// one sequence (append, fold, which checkpoint copy to read), the pointer
// update that the last reader of a sequence performs, and the bounded
// mbarrier wait.  The record window and the pointer rules are those of
// "ReplaySSM: Cache SSM Inputs, Not State", section "How it works": h records
// since the checkpoint at slots base .. base+h-1 (mod capacity), a fold when
// the window fills, and speculative drafts that stay uncommitted (nd) until
// commit or rollback move the pointers.
#pragma once

#include "rs_common.cuh"
#include "rs_internal.h"

namespace rs {

// What one launch does to one sequence, from its pointers and the mode.
struct SeqPlan {
    int base, hc, ndr;
    int T;       // records appended by this launch
    int F;       // records folded into the checkpoint (0: none)
    int fold, ok, append, work;
    unsigned err;
};

__device__ __forceinline__ SeqPlan plan_sequence(const ReplayParams &p, int b) {
    SeqPlan s;
    const int mode = p.mode, cap = p.cap, L = p.L;
    s.base = p.base[b];
    s.hc = p.h[b];
    s.ndr = p.nd[b];
    s.T = mode == MODE_DECODE ? 1 : (mode == MODE_VERIFY ? p.T : 0);
    s.F = 0;
    s.fold = 0;
    s.append = 0;
    s.err = 0;
    // a pointer state outside the buffer (never produced by the library) is
    // reported and the sequence left untouched rather than indexed with it
    s.ok = s.base >= 0 && s.base < cap && s.hc >= 0 && s.hc <= cap && s.ndr >= 0 && s.ndr <= cap;
    if (s.ok) {
        if (mode == MODE_DECODE) {
            if (s.ndr) s.err |= RS_DEV_DRAFTS_PENDING;
            s.ok = s.hc + 1 <= cap;
            s.F = s.hc + 1;
            s.fold = s.F >= L;
            s.append = !s.fold;  // a folded record never needs its buffer slot
        } else if (mode == MODE_VERIFY) {
            if (s.ndr) s.err |= RS_DEV_DRAFTS_PENDING;
            s.ok = s.hc + s.T <= cap;
            s.fold = s.hc + s.T > L && s.hc > 0;
            s.F = s.fold ? s.hc : 0;
            s.append = 1;
        } else {  // flush / materialise: the committed records
            s.F = s.hc;
            s.fold = mode == MODE_FLUSH && s.hc > 0;
        }
    }
    if (!s.ok) s.err |= RS_DEV_CAPACITY;
    s.work = s.ok && (mode != MODE_FLUSH || s.fold);
    return s;
}

// Called once per unit, by the thread that read the unit's pointers.  The
// counter's address depends on the values read, so the increment cannot be
// performed before those reads completed; the unit that sees the count reach
// units_per_seq-1 is the last reader of sequence b and writes the new
// pointers at once.  atomicInc wraps the counter back to 0 for the next launch.
__device__ __forceinline__ void arrive_and_update(const ReplayParams &p, const SeqPlan &s, int b,
                                                  unsigned units_per_seq, bool report) {
    if (p.mode == MODE_MATERIALIZE) return;
    if (report && s.err) atomicOr(p.status, s.err);
    const unsigned z = zero_dependent_on((unsigned)(s.base ^ s.hc ^ s.ndr));
    const unsigned prev = atomicInc(p.arrive + b + z, units_per_seq - 1);
    if (prev != units_per_seq - 1 || !s.ok) return;
    const int cap = p.cap;
    if (p.mode == MODE_DECODE) {
        if (s.fold) { p.base[b] = (s.base + s.F) % cap; p.h[b] = 0; }
        else p.h[b] = s.hc + 1;
        p.nd[b] = 0;
    } else if (p.mode == MODE_VERIFY) {
        if (s.fold) { p.base[b] = (s.base + s.hc) % cap; p.h[b] = 0; }
        p.nd[b] = s.T;
    } else if (s.fold) {  // flush
        p.base[b] = (s.base + s.hc) % cap;
        p.h[b] = 0;
    }
}

// Dynamic unit scheduling (the row-split pipeline).  A launch's units are
// handed out in order from one counter, arrive[B]: each CTA takes its next
// unit when its producer is ready to plan one, so that a CTA that drew costly
// units (a folding unit moves twice the bytes of a streamed one, and which
// sequences fold depends on their pointers) takes fewer.  The producers finish
// by counting themselves on arrive[B + 1]; the last one resets both counters
// for the next launch on the state.  (Mamba-2 decode 0.1844 against 0.1876 ms
// per step with round-robin units, its 4-draft round 0.303 against 0.316 ms.)
__device__ __forceinline__ int next_unit(const ReplayParams &p) {
    return (int)atomicAdd(p.arrive + p.B, 1u);
}
__device__ __forceinline__ void planner_done(const ReplayParams &p, unsigned planners) {
    uint32_t *ctr = p.arrive + p.B;
    if (atomicAdd(ctr + 1, 1u) == planners - 1) {
        ctr[0] = 0u;
        ctr[1] = 0u;
    }
}

// Two-precision: a folding sequence reads the fp32 copy, any other the bf16
// copy; shared-bf16 has only the bf16 copy.
__device__ __forceinline__ bool plan_reads_lp(const ReplayParams &p, const SeqPlan &s) {
    return p.prec == RS_PREC_SHARED_BF16 ||
           (p.prec == RS_PREC_TWO && !s.fold && (p.mode == MODE_DECODE || p.mode == MODE_VERIFY));
}

// mbarrier wait that also gives up as soon as another role of the CTA has
// aborted (the flag lives in shared memory).
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, unsigned parity, volatile int *abort_flag,
                                              uint32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity)) {
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(status, RS_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

}  // namespace rs
