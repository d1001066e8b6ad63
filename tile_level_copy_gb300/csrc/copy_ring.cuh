// Row-band copy engine of the return path: Yp rows -> the owner's slice of Ret.
//
// "Fine-grained Computation-Communication Overlap via Tile-level Signaling and Scheduling for
// Mixture-of-Experts" (pith.science/paper/W2ZARMHG), "Core claim": the consumer polls the tile
// flags and issues one contiguous write per row-band segment. On one GPU the write is an
// HBM-to-HBM copy; each CTA moves it through a ring of shared-memory buffers with TMA bulk copies
// (global -> shared completes on an mbarrier, shared -> global is a bulk group), so one thread
// keeps up to COPY_NBUF * COPY_PIECE bytes in flight.
//
// Work units: band (schedule position) x row chunk of rows_per_unit rows, handed out in schedule
// order by an atomic counter, so idle CTAs always take the oldest outstanding band.
#pragma once

#include "moe_internal.cuh"

namespace moe {

struct CopyRing {
    uint8_t* buf;         // COPY_NBUF buffers of COPY_PIECE bytes, 1024-byte aligned
    uint64_t* bar;        // COPY_NBUF mbarriers, count 1
    uint32_t phase_bits;  // parity to wait for next, per buffer
    uint32_t pending;     // buffers with a load in flight that has not been waited for
};

// Thread-0 only. Copies `bytes` (multiple of 16) from src to dst. Returns false on timeout.
__device__ __forceinline__ bool ring_copy(CopyRing& cr, const uint8_t* src, uint8_t* dst, size_t bytes,
                                          unsigned long long timeout_ns, volatile int* abort) {
    const int np = (int)((bytes + COPY_PIECE - 1) / COPY_PIECE);
    bulk_wait_read_all();  // every earlier store has finished reading its buffer
    auto issue = [&](int i) {
        const int b = i % COPY_NBUF;
        const uint32_t len = (uint32_t)min((size_t)COPY_PIECE, bytes - (size_t)i * COPY_PIECE);
        mbar_arrive_expect_tx(&cr.bar[b], len);
        bulk_load(cr.buf + (size_t)b * COPY_PIECE, src + (size_t)i * COPY_PIECE, len, &cr.bar[b]);
        cr.pending |= 1u << b;
    };
    const int pro = min(np, COPY_NBUF);
    for (int i = 0; i < pro; ++i) issue(i);
    for (int i = 0; i < np; ++i) {
        const int b = i % COPY_NBUF;
        if (!mbar_wait(&cr.bar[b], (cr.phase_bits >> b) & 1u, timeout_ns, abort)) return false;
        cr.phase_bits ^= 1u << b;
        cr.pending &= ~(1u << b);
        const uint32_t len = (uint32_t)min((size_t)COPY_PIECE, bytes - (size_t)i * COPY_PIECE);
        bulk_store(dst + (size_t)i * COPY_PIECE, cr.buf + (size_t)b * COPY_PIECE, len);
        bulk_commit();
        if (i + COPY_NBUF < np) {
            bulk_wait_read_all();
            issue(i + COPY_NBUF);
        }
    }
    return true;
}

// Before the CTA leaves: wait (bounded) for loads still in flight, then for all stores.
__device__ __forceinline__ void ring_drain(CopyRing& cr, unsigned long long timeout_ns) {
    int never = 0;
    for (int b = 0; b < COPY_NBUF; ++b)
        if (cr.pending & (1u << b)) {
            mbar_wait(&cr.bar[b], (cr.phase_bits >> b) & 1u, timeout_ns, &never);
            cr.phase_bits ^= 1u << b;
        }
    cr.pending = 0;
    bulk_wait_all();
}

// All threads of the CTA call this. Takes units from meta[queue] until none is left.
// wait_flags: acquire every tile flag of the unit's segment (== want) before copying.
__device__ void copy_units(const Shape& s, const PlanPtrs& p, CopyRing& cr, volatile int* s_unit,
                           volatile int* s_abort, int queue, bool wait_flags, uint32_t want) {
    const int tid = threadIdx.x;
    int MT = p.meta[META_MTILES];
    if (MT < 0 || MT > s.MT_max) MT = 0;
    const int units = MT * s.units_per_band;
    const size_t rowb = (size_t)s.d * 2;
    unsigned long long t_first = ~0ull;
    bool did = false;

    for (;;) {
        if (tid == 0) *s_unit = atomicAdd(&p.meta[queue], 1);
        __syncthreads();
        const int u = *s_unit;
        const bool stop = *s_abort != 0;
        __syncthreads();
        if (u >= units || stop) break;
        const int pos = u / s.units_per_band, c = u % s.units_per_band;
        const int m = p.sched[pos];
        const int row0 = p.tiles[4 * m + 2], valid = p.tiles[4 * m + 3];
        const int rb = c * s.rows_per_unit;
        if (rb >= valid) continue;
        const int re = min(valid, rb + s.rows_per_unit);

        if (wait_flags) {
            const int first = p.seg[2 * pos], nb = p.seg[2 * pos + 1];
            const int nf = nb * s.n_tiles_n2;
            if (tid < nf) {
                const int mb = p.sched[first + tid / s.n_tiles_n2];
                const uint32_t* f = p.flags + (size_t)mb * s.n_tiles_n2 + (tid % s.n_tiles_n2);
                if (ld_acquire_gpu(f) != want) {
                    const unsigned long long t0 = globaltimer();
                    for (;;) {
                        __nanosleep(40);
                        if (ld_acquire_gpu(f) == want) break;
                        if (*s_abort) break;
                        if (globaltimer() - t0 > s.timeout_ns) {
                            *s_abort = 1;
                            set_status(p.meta, ST_FLAG_TIMEOUT, mb);
                            break;
                        }
                    }
                }
            }
            __syncthreads();
            if (*s_abort) break;
        }
        if (tid == 0) {
            if (!did) t_first = globaltimer();
            did = true;
            fence_proxy_async_global();
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.Yp) + (size_t)(row0 + rb) * rowb;
            uint8_t* dst = reinterpret_cast<uint8_t*>(p.Ret) + (size_t)(p.tile_ret[m] + rb) * rowb;
            if (!ring_copy(cr, src, dst, (size_t)(re - rb) * rowb, s.timeout_ns, s_abort)) {
                *s_abort = 1;
                set_status(p.meta, ST_COPY_TIMEOUT, m);
            }
        }
    }
    if (tid == 0) {
        ring_drain(cr, s.timeout_ns);
        if (did) {
            atomicMin(&p.trace[MOE_TRACE_COPY_START], t_first);
            atomicMax(&p.trace[MOE_TRACE_COPY_END], globaltimer());
        }
    }
    __syncthreads();
}

}  // namespace moe
