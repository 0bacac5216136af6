// Streaming scheduler (see ls_sched.h for the rules it implements).
#include "ls_sched.h"

#include <algorithm>

namespace ls {

static inline int64_t align256(int64_t n) { return (n + 255) / 256 * 256; }

Plan make_plan(int N, int64_t S, int64_t shared_total, int depth, int resident, int64_t max_vram,
               int slot_cap) {
    Plan p;
    p.N = N;
    p.S = S;
    p.shared_total = shared_total;
    int avail;
    if (max_vram == 0) {
        if (slot_cap < 0) {  // segmentation off: all resident, controls have no effect
            p.avail = N;
            p.d_fit = 0;
            p.R = N;
            p.Q = 0;
            p.P = N;
            return p;
        }
        avail = N;
    } else {
        int64_t room = max_vram - shared_total;
        int64_t a = room > 0 ? room / S : 0;
        if (a < 1) {  // the mandatory execution slot only
            p.avail = 1;
            p.d_fit = 0;
            p.R = 0;
            p.Q = 1;
            p.P = 1;
            p.mandatory = true;
            return p;
        }
        avail = (int)std::min<int64_t>(a, 1 << 30);
    }
    if (slot_cap >= 0) avail = std::min(avail, slot_cap);
    p.avail = avail;
    // depth first: with no residents the ring of d+1 slots (at most N) must fit
    int d_fit = avail >= N ? depth : std::min(depth, avail - 1);
    int cap = resident < 0 ? N : std::min(resident, N);
    int R = 0;
    for (int r = cap; r >= 0; --r) {
        int64_t need = std::min<int64_t>((int64_t)r + d_fit + 1, N);
        if (need <= avail) {
            R = r;
            break;
        }
    }
    int M = N - R;
    p.d_fit = d_fit;
    p.R = R;
    p.Q = M > 0 ? std::min(d_fit + 1, M) : 0;
    p.P = R + p.Q;
    return p;
}

void Scheduler::configure(const ls_params& p, const std::vector<int64_t>& seg_slot,
                          const std::vector<std::pair<int, int64_t>>& shared) {
    prm_ = p;
    seg_slot_ = seg_slot;
    shared_ = shared;
    std::sort(shared_.begin(), shared_.end());
    cap_ = p.test_alloc_cap_bytes;
    fail_async_ = p.test_fail_async != 0;
    cross_run_ = p.cross_run_prefetch != 0;
}

void Scheduler::emit(int step, int kind, int seg, int slot, int64_t bytes) {
    ls_sched_event e{};
    e.run = run_;
    e.step = step;
    e.kind = kind;
    e.segment = seg;
    e.slot = slot;
    e.bytes = bytes;
    log_.push_back(e);
}

void Scheduler::fallback() {
    async_ok_ = false;
    fail_async_ = false;
    d_ = 0;
    ++n_fallback;
    warnings |= 1 << LS_WARN_SYNC_FALLBACK;
}

ls_status Scheduler::register_memory(Executor& ex) {
    const int N = (int)seg_slot_.size();
    int64_t S = 0;
    for (int64_t b : seg_slot_) S = std::max(S, b);
    int64_t shared_total = 0;
    for (auto& s : shared_) shared_total += align256(s.second);
    Plan p = make_plan(N, S, shared_total, prm_.prefetch_depth, prm_.resident_layers,
                       prm_.max_vram_bytes, -1);
    const bool mandatory = p.mandatory;
    if (mandatory) warnings |= 1 << LS_WARN_MANDATORY_SLOT;
    if (shared_total > 0) {
        if (!alloc_bytes(shared_total)) return LS_ERR_OOM;
        if (!ex.alloc_shared(shared_total)) {
            live_ -= shared_total;
            return LS_ERR_OOM;
        }
    }
    if (prm_.use_pool && !alloc_pool_degrading(ex, p)) return LS_ERR_OOM;
    plan_ = p;
    R_ = p.R;
    d_ = p.d_fit;
    loaded_R_ = 0;
    return mandatory ? LS_WARN_MANDATORY_SLOT : LS_OK;
}

// The pool for plan p, or for fewer slots of the same size (re-planned for that many) when
// the allocation fails; a reduced count is remembered for later plans. p becomes the plan
// that got its pool.
bool Scheduler::alloc_pool_degrading(Executor& ex, Plan& p) {
    const bool mandatory = p.mandatory;
    for (int cap = p.P; cap >= 1; --cap) {
        Plan q = cap == p.P ? p
                            : make_plan(p.N, p.S, p.shared_total, prm_.prefetch_depth, prm_.resident_layers,
                                        prm_.max_vram_bytes, cap);
        q.mandatory = mandatory;
        const int64_t bytes = (int64_t)q.P * q.S;
        if (alloc_bytes(bytes)) {
            if (ex.alloc_pool(q.P, q.S)) {
                if (q.P < p.P) slot_cap_ = q.P;
                p = q;
                return true;
            }
            live_ -= bytes;
        }
        ++n_degrade;
    }
    return false;
}

void Scheduler::release_carried(Executor& ex) {
    for (auto& cs : carried_) {
        emit(-1, LS_EV_EVICT, cs.first, cs.second, 0);
        ++n_evict;
        ex.evict(cs.first, cs.second);
        if (!prm_.use_pool) live_ -= seg_slot_[cs.first];
    }
    carried_.clear();
}

void Scheduler::evict_residents_down_to(Executor& ex, int keep) {
    for (int r = loaded_R_ - 1; r >= keep; --r) {
        emit(-1, LS_EV_EVICT, r, r, 0);
        ++n_evict;
        ex.evict(r, r);
        if (!prm_.use_pool) live_ -= seg_slot_[r];
    }
    loaded_R_ = std::min(loaded_R_, keep);
}

ls_status Scheduler::replan(Executor& ex, int depth, int resident, int64_t max_vram) {
    if (!usable_) return LS_ERR_STATE;
    prm_.prefetch_depth = depth;
    prm_.resident_layers = resident;
    prm_.max_vram_bytes = max_vram;
    release_carried(ex);
    Plan p = make_plan(plan_.N, plan_.S, plan_.shared_total, depth, resident, max_vram, slot_cap_);
    const bool mandatory = p.mandatory;
    if (prm_.use_pool && p.P != plan_.P) {
        // another slot count: the pool is given back first, so every slot empties
        evict_residents_down_to(ex, 0);
        ex.free_pool();
        live_ -= (int64_t)plan_.P * plan_.S;
        if (!alloc_pool_degrading(ex, p)) {
            usable_ = false;
            return LS_ERR_OOM;
        }
    } else {
        evict_residents_down_to(ex, p.R);  // stale residents, from the end of the prefix
    }
    plan_ = p;
    R_ = p.R;  // a grown prefix is allocated and loaded at the next run
    loaded_R_ = std::min(loaded_R_, p.R);
    d_ = async_ok_ ? p.d_fit : 0;
    J_ = 0;
    if (mandatory) warnings |= 1 << LS_WARN_MANDATORY_SLOT;
    return mandatory ? LS_WARN_MANDATORY_SLOT : LS_OK;
}

bool Scheduler::alloc_seg_evicting(Executor& ex, int seg, int step, int& cur_R) {
    for (;;) {
        if (alloc_bytes(seg_slot_[seg])) {
            if (ex.alloc_segment(seg, seg_slot_[seg])) return true;
            live_ -= seg_slot_[seg];
        }
        int r = cur_R - 1;
        if (r < 0 || r >= step) return false;  // never the active one, never one not yet computed
        emit(step, LS_EV_EVICT, r, r, 0);
        ++n_evict;
        ex.evict(r, r);
        live_ -= seg_slot_[r];
        cur_R = r;
    }
}

ls_status Scheduler::run(Executor& ex, const int64_t* load_bytes) {
    if (!usable_) return LS_ERR_STATE;
    const int N = plan_.N;
    const bool pool = prm_.use_pool != 0;
    auto lb = [&](int s) { return load_bytes ? load_bytes[s] : seg_slot_[s]; };
    ex.begin_run(run_);
    if (run_ == 0) {
        for (auto& s : shared_) {
            emit(-1, LS_EV_SHARED_LOAD, s.first, -1, s.second);
            ex.load_shared(s.first);
            ++n_shared;
            bytes_loaded += s.second;
        }
    }
    if (!carried_.empty() && carried_R_ != R_) release_carried(ex);  // planned for another ring
    for (int i = loaded_R_; i < R_; ++i) {  // residents that hold no data yet
        if (!pool) {
            if (!alloc_bytes(seg_slot_[i])) {
                R_ = i;
                break;
            }
            if (!ex.alloc_segment(i, seg_slot_[i])) {
                live_ -= seg_slot_[i];
                R_ = i;
                break;
            }
        }
        emit(-1, LS_EV_LOAD_RESIDENT, i, i, lb(i));
        ex.load(i, i, LS_EV_LOAD_RESIDENT, lb(i));
        ++n_resident;
        bytes_loaded += lb(i);
    }
    loaded_R_ = R_;
    const int R = R_;
    const int M = N - R;
    const int Q = M > 0 ? std::min(d_ + 1, M) : 0;
    int d = std::min(d_, M);
    const int64_t J0 = cross_run_ ? J_ : 0;
    // the window reaches into the next run only with a full ring of d + 1 slots
    const int reach = (cross_run_ && M > d) ? M + d : M;
    auto ring_slot = [&](int64_t j) { return R + (int)((J0 + j) % Q); };
    int cur_R = R;
    std::vector<char> queued(N, 0);
    for (auto& cs : carried_) queued[cs.first] = 1;  // issued by the previous run
    int next_load = (int)carried_.size();
    carried_.clear();
    bool fell_back = false;
    ls_status st = LS_OK;
    for (int k = 0; k < N; ++k) {
        const int streamed_upto = std::max(0, k - R + 1);
        if (d >= 1 && async_ok_) {
            while (next_load < reach && next_load < streamed_upto + d) {
                const int seg = R + next_load % M;
                if (next_load >= M) {
                    // the next run's loads never evict: without room that run loads them itself
                    if (!pool) {
                        if (!alloc_bytes(seg_slot_[seg])) break;
                        if (!ex.alloc_segment(seg, seg_slot_[seg])) {
                            live_ -= seg_slot_[seg];
                            break;
                        }
                    }
                } else if (fail_async_ || (!pool && !alloc_seg_evicting(ex, seg, k, cur_R))) {
                    fallback();
                    fell_back = true;
                    d = 0;
                    break;
                }
                const int slot = ring_slot(next_load);
                emit(k, LS_EV_PREFETCH, seg, slot, lb(seg));
                ex.load(seg, slot, LS_EV_PREFETCH, lb(seg));
                ++n_prefetch;
                bytes_loaded += lb(seg);
                if (next_load < M)
                    queued[seg] = 1;
                else
                    carried_.push_back({seg, slot});
                ++next_load;
            }
        }
        if (k >= R && !queued[k]) {
            if (!pool && !alloc_seg_evicting(ex, k, k, cur_R)) {
                st = LS_ERR_OOM;
                break;
            }
            const int slot = ring_slot(k - R);
            emit(k, LS_EV_LOAD_SYNC, k, slot, lb(k));
            ex.load(k, slot, LS_EV_LOAD_SYNC, lb(k));
            ++n_sync;
            bytes_loaded += lb(k);
            next_load = k - R + 1;
        }
        const int slot = k < R ? k : ring_slot(k - R);
        emit(k, LS_EV_ACTIVATE, k, slot, 0);
        ex.activate(k, slot, queued[k] != 0);
        if (queued[k]) ++n_prefetch_activated;
        if (!pool && k >= R) {
            ex.free_segment(k);
            live_ -= seg_slot_[k];
        }
    }
    R_ = cur_R;
    loaded_R_ = std::min(loaded_R_, R_);
    carried_R_ = R;
    if (cross_run_) J_ = J0 + M;
    ++run_;
    if (st != LS_OK) return st;
    return fell_back ? LS_WARN_SYNC_FALLBACK : LS_OK;
}

void Scheduler::fill_stats(ls_stats& s) const {
    s.n_segments = plan_.N;
    s.residents = R_;
    int M = plan_.N - R_;
    s.depth = std::min(d_, M);
    s.ring_slots = M > 0 ? std::min(d_ + 1, M) : 0;
    s.pool_slots = plan_.P;
    s.warnings = warnings;
    s.slot_bytes = plan_.S;
    s.shared_bytes = plan_.shared_total;
    s.pool_bytes = prm_.use_pool ? (int64_t)plan_.P * plan_.S : 0;
    s.runs = run_;
    s.prefetch_queued = n_prefetch;
    s.prefetch_activated = n_prefetch_activated;
    s.sync_loads = n_sync;
    s.resident_loads = n_resident;
    s.shared_loads = n_shared;
    s.evictions = n_evict;
    s.sync_fallbacks = n_fallback;
    s.pool_degradations = n_degrade;
    s.bytes_loaded = bytes_loaded;
}

}  // namespace ls
