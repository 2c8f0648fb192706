// unit_ring.cuh -- work units claimed in order for persistent (pair) kernels.
//
// The producer thread of a cluster's even CTA claims the next unit from one
// grid-wide counter (zeroed before the launch) and hands it to every other role
// of the cluster -- its own CTA's UMMA issuer and epilogue warps, and in a CTA
// pair the odd CTA's producer and epilogue warps -- through a ring of
// shared-memory slots guarded by mbarriers.  So the units in flight across the
// grid always form one window of consecutive indices however the clusters'
// speeds differ, and the operand tiles they share are read from HBM once, then
// from L2.  Which cluster runs a unit never changes a result bit.
//
// A slot holds a unit index or -1 (no unit left).  The claiming producer
// publishes one unit ahead of its own loads; a slot is reused once every role
// has read it, so with units of many k-steps (roles at most two units behind:
// two TMEM accumulators) the producer never waits for one, and with units of
// a few k-steps the four slots, not the stage ring, bound how far it runs
// ahead.  Every wait is bounded.
#pragma once

#include <cstdint>

#include "tim_ptx.cuh"

namespace tim {

constexpr int UNIT_RING_SLOTS = 4;
constexpr uint32_t UNIT_RING_BYTES = UNIT_RING_SLOTS * (2 * 8 + 4);   // two mbarriers and a word per slot

// CL: CTAs per cluster (1 or 2); USERS: roles that take each unit (they release the slot).
template <int CL, uint32_t USERS>
struct UnitRing {
    uint32_t bar0;              // shared::cta address of the 2 x SLOTS mbarriers (full, then empty)
    volatile int32_t *unit;     // the slots
    int slot = 0;
    uint32_t phase = 0;

    // `base`: UNIT_RING_BYTES of shared memory, 8-byte aligned.
    __device__ explicit UnitRing(uint8_t *base)
        : bar0(smem_u32(base)), unit(reinterpret_cast<volatile int32_t *>(base + UNIT_RING_SLOTS * 16)) {}

    __device__ uint32_t full(int i) const { return bar0 + 8u * i; }
    __device__ uint32_t empty(int i) const { return bar0 + 8u * (UNIT_RING_SLOTS + i); }

    // One thread per CTA, before the cluster barrier that precedes any use.
    __device__ void init() const
    {
        for (int i = 0; i < UNIT_RING_SLOTS; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), USERS);   // in a pair only the even CTA's counts
        }
    }

    __device__ void advance()
    {
        if (++slot == UNIT_RING_SLOTS) {
            slot = 0;
            phase ^= 1u;
        }
    }

    // The even CTA's producer: claims the next unit (or -1 past `units`) and
    // publishes it to both CTAs.  false when a wait ran out of time.
    __device__ bool claim(int *counter, int units, int &u, volatile int *abort, uint64_t budget)
    {
        if (!mbar_wait(empty(slot), phase ^ 1u, abort, budget))
            return false;
        u = atomicAdd(counter, 1);
        if (u >= units)
            u = -1;
        unit[slot] = u;
        if (CL == 2) {   // the odd CTA's copy of the slot, then its barrier (release at cluster scope)
            st_shared_cluster(mapa_shared(smem_u32(const_cast<int32_t *>(unit + slot)), 1), u);
            mbar_arrive_remote(mapa_shared(full(slot), 1));
        }
        mbar_arrive(full(slot));
        advance();
        return true;
    }

    // The even CTA's producer, one unit ahead: returns in `u` the unit to load
    // now (claimed and published earlier, in `ahead`; -1 when none is left) and
    // claims the one after it, so the counter's latency overlaps this unit's
    // loads.  Start with claim(counter, units, ahead, ...).
    __device__ bool next(int *counter, int units, int &u, int &ahead, volatile int *abort, uint64_t budget)
    {
        u = ahead;
        return u < 0 || claim(counter, units, ahead, abort, budget);
    }

    // Any other role: the next unit.  `arrive` (one lane per role) releases the
    // slot, on the even CTA's barrier, once the unit has been read.
    __device__ bool take(int &u, bool arrive, uint32_t rank, volatile int *abort, uint64_t budget)
    {
        const bool got = rank == 0 ? mbar_wait(full(slot), phase, abort, budget)
                                   : mbar_wait_cluster(full(slot), phase, abort, budget);
        if (!got)
            return false;
        u = unit[slot];
        __syncwarp(__activemask());
        if (arrive) {
            if (CL == 2)
                mbar_arrive_remote_cta(mapa_shared(empty(slot), 0));
            else
                mbar_arrive(empty(slot));
        }
        advance();
        return true;
    }
};

} // namespace tim
