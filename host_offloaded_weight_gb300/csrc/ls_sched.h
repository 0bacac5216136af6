// Streaming scheduler: slot plan, prefetch window, resident prefix, pool
// degradation, synchronous fallback, eviction. Host-only integer logic.
//
// Rules ("feat: prefetch streamed layers during compute", Summary and Effective
// behavior table; "feat: pool VRAM for streamed layer", Summary and pool
// behavior table):
//   S  = largest 256-byte-aligned private footprint of a segment.
//   max_vram_bytes == 0: segmentation off, every segment resident.
//   otherwise avail = floor((budget - shared) / S); below one slot the single
//   mandatory slot is taken with a warning and nothing else (no residents, no
//   prefetch).
//   Depth first: the largest depth <= requested whose ring fits with no
//   residents; then the longest resident prefix <= cap that still fits.
//   Ring Q = min(d + 1, N - R); pool P = R + Q. Load j of a run goes to slot
//   R + (j mod Q); resident i lives in slot i.
//   Per step k: queue prefetches until the loads issued reach (streamed
//   segments <= k) + d; load k synchronously if it was not queued; activate k.
//   A failing pool is retried with fewer slots of the same size (re-planned
//   for that many, and the reduced count is remembered); pool off, a failing
//   load first evicts the last resident already computed in this run, a
//   failing prefetch then falls back to synchronous loads for good, a failing
//   synchronous load fails the run.
// Plan changes between runs (replan): prefetches issued for the next run are
//   released, residents the new plan does not hold are released from the end of
//   the prefix; the pool is kept at the same slot count and reallocated
//   otherwise (emptying every slot); each run first loads the residents that
//   hold no data yet. Cross-run window (opt-in): the window of the last steps
//   reaches into the next run's first streamed segments when the ring is a full
//   d + 1 slots; load numbers then continue across runs (slot R + (J mod Q)).
#pragma once
#include <cstdint>
#include <vector>

#include "ls_api.h"

namespace ls {

struct Plan {
    int N = 0;
    int64_t S = 0;
    int64_t shared_total = 0;
    int avail = 0;
    int d_fit = 0;   // depth that fits, before capping by the streamed count
    int R = 0;
    int Q = 0;
    int P = 0;
    bool mandatory = false;
};

Plan make_plan(int N, int64_t S, int64_t shared_total, int depth, int resident, int64_t max_vram,
               int slot_cap /* < 0: none */);

// What the scheduler asks of the device side. Every call is made in schedule
// order; a false return from an allocation means the memory is not available.
struct Executor {
    virtual ~Executor() {}
    virtual bool alloc_shared(int64_t bytes) = 0;
    virtual bool alloc_pool(int slots, int64_t slot_bytes) = 0;
    virtual bool alloc_segment(int seg, int64_t bytes) = 0;   // pool off: one buffer per load/resident
    virtual void free_segment(int seg) = 0;                    // ordered after the segment's compute
    virtual void begin_run(int run) = 0;
    virtual void load_shared(int shared_id) = 0;
    virtual void load(int seg, int slot, int kind, int64_t bytes) = 0;   // kind = LS_EV_*
    virtual void activate(int seg, int slot, bool via_copy_queue) = 0;
    virtual void evict(int seg, int slot) = 0;              // resident, or a stale prefetch
    virtual void free_pool() = 0;                           // before a pool of another size
};

class Scheduler {
public:
    // seg_slot: aligned private footprint per segment; shared: (id, bytes) distinct ids.
    void configure(const ls_params& p, const std::vector<int64_t>& seg_slot,
                   const std::vector<std::pair<int, int64_t>>& shared);
    ls_status register_memory(Executor& ex);                 // plan + shared region + pool
    ls_status run(Executor& ex, const int64_t* load_bytes);  // one pass; load_bytes[N] or null
    // New controls for the next run; LS_ERR_OOM (no pool at all) leaves the scheduler unusable.
    ls_status replan(Executor& ex, int depth, int resident, int64_t max_vram);
    bool usable() const { return usable_; }
    const Plan& plan() const { return plan_; }
    const std::vector<ls_sched_event>& log() const { return log_; }
    // A copy of the scheduler state without the event log (to predict a run cheaply).
    Scheduler without_log() {
        std::vector<ls_sched_event> keep;
        keep.swap(log_);
        Scheduler copy = *this;
        log_.swap(keep);
        return copy;
    }
    void fill_stats(ls_stats& s) const;
    int residents() const { return R_; }
    int depth() const { return d_; }
    int runs() const { return run_; }
    int64_t live_bytes() const { return live_; }

private:
    bool alloc_bytes(int64_t bytes) {
        if (cap_ > 0 && live_ + bytes > cap_) return false;
        live_ += bytes;
        return true;
    }
    bool alloc_seg_evicting(Executor& ex, int seg, int step, int& cur_R);
    bool alloc_pool_degrading(Executor& ex, Plan& p);
    void release_carried(Executor& ex);
    void evict_residents_down_to(Executor& ex, int keep);
    void emit(int step, int kind, int seg, int slot, int64_t bytes);
    void fallback();

    ls_params prm_{};
    std::vector<int64_t> seg_slot_;
    std::vector<std::pair<int, int64_t>> shared_;
    Plan plan_;
    int R_ = 0, d_ = 0, run_ = 0;
    bool async_ok_ = true, fail_async_ = false, cross_run_ = false, usable_ = true;
    int slot_cap_ = -1;                            // remembered reduced pool slot count
    int loaded_R_ = 0;                             // leading residents holding their data
    int64_t J_ = 0;                                // streamed loads since the last plan change
    std::vector<std::pair<int, int>> carried_;     // (segment, slot) prefetched for the next run
    int carried_R_ = 0;
    int64_t cap_ = 0, live_ = 0;
    std::vector<ls_sched_event> log_;

public:
    int64_t n_prefetch = 0, n_prefetch_activated = 0, n_sync = 0, n_resident = 0,
            n_shared = 0, n_evict = 0, n_fallback = 0, n_degrade = 0, bytes_loaded = 0;
    int warnings = 0;
};

}  // namespace ls
