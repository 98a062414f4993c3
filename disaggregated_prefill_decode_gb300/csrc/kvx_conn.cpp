// Host-side connector state machine around the push: rendezvous of the consumer's registration and
// the producer's prefill, chunked-prefill gating, deferral with a timeout, sealed write counts per
// producer rank, batch-state decision for each write and load errors. No CUDA call: every call takes
// the caller's clock, so the protocol runs (and is tested) on any host.
//
// Follows the push-mode NIXL connector article (spke.com 3844), "Implementierungsdetails" steps 1-3,
// and the "vLLM MoRIIO KV Connector" notes, sections 3.1, 3.2, 5 and 6 (which facts come from where
// is listed beside the declarations in kvx.h).
#include "kvx_internal.h"

#include <algorithm>
#include <deque>
#include <map>
#include <mutex>
#include <new>
#include <unordered_map>

namespace kvx {

struct ConnRank {
    int64_t issued = 0;
    int64_t expected = -1;        // -1 until the rank seals
    int64_t done = 0;             // writes reported, failed ones included
};

struct ConnRecord {
    uint64_t serial = 0;          // changes whenever the record starts over; stale deadlines/events carry an old one
    int32_t attempt = 0;
    int32_t state = KVX_CONN_WAITING;
    bool registered = false;
    bool prefill_done = false;
    int32_t n_chunks = 0;
    int64_t n_tokens = 0;
    std::vector<int32_t> src, dst;
    std::vector<ConnRank> ranks;
    int64_t writes_failed = 0;
    std::vector<int32_t> load_errors;   // distinct consumer block ids, in the order first reported
};

enum DeadlineKind { kDefer, kTransfer, kAbort };

struct Deadline {
    int64_t req_id;
    uint64_t serial;
    DeadlineKind kind;
};

struct ConnEvent {
    int64_t req_id;
    uint64_t serial;
    int32_t attempt;
    int32_t state;
};

}  // namespace kvx

struct kvx_conn_s {
    kvx_conn_config cfg{};
    std::mutex mu;
    uint64_t next_serial = 1;
    std::unordered_map<int64_t, kvx::ConnRecord> recs;
    std::multimap<int64_t, kvx::Deadline> deadlines;   // by due time; equal times keep insertion order
    std::deque<kvx::ConnEvent> events;
};

using namespace kvx;

namespace {

constexpr int64_t kSecond = 1000 * 1000;
constexpr int32_t kMaxRanks = 1 << 16;   // every record keeps one counter set per rank

bool terminal(int32_t s) {
    return s == KVX_CONN_DONE || s == KVX_CONN_FAILED || s == KVX_CONN_EXPIRED || s == KVX_CONN_TIMED_OUT ||
           s == KVX_CONN_ABORTED;
}

void emit(kvx_conn_s *k, int64_t id, const ConnRecord &r) {
    k->events.push_back(ConnEvent{id, r.serial, r.attempt, r.state});
}

void add_deadline(kvx_conn_s *k, int64_t due, int64_t id, const ConnRecord &r, DeadlineKind kind) {
    k->deadlines.emplace(due, Deadline{id, r.serial, kind});
}

void start_over(kvx_conn_s *k, ConnRecord &r, int32_t attempt) {
    r = ConnRecord();
    r.serial = k->next_serial++;
    r.attempt = attempt;
    r.ranks.resize(k->cfg.n_ranks);
}

// The record for (id, attempt): nullptr for a stale attempt, a fresh record for a newer one.
ConnRecord *record_for(kvx_conn_s *k, int64_t id, int32_t attempt) {
    auto it = k->recs.find(id);
    if (it == k->recs.end()) {
        ConnRecord &r = k->recs[id];
        start_over(k, r, attempt);
        return &r;
    }
    ConnRecord &r = it->second;
    if (attempt < r.attempt) return nullptr;
    if (attempt > r.attempt) start_over(k, r, attempt);              // retried or preempted request
    return &r;
}

// Rendezvous: whichever of registration and last prefill chunk comes second makes the record READY.
void rendezvous(kvx_conn_s *k, int64_t id, ConnRecord &r, int64_t now) {
    if (r.state != KVX_CONN_WAITING && r.state != KVX_CONN_DEFERRED) return;
    if (r.registered && r.prefill_done) {
        r.state = KVX_CONN_READY;
        emit(k, id, r);
    } else if (r.prefill_done && r.state == KVX_CONN_WAITING) {
        r.state = KVX_CONN_DEFERRED;                                  // the producer holds its blocks
        add_deadline(k, now + k->cfg.defer_timeout_us, id, r, kDefer);
    }
}

// IN_FLIGHT -> DONE / FAILED once every rank sealed and reported every write it queued.
void complete_if_counted(kvx_conn_s *k, int64_t id, ConnRecord &r) {
    if (r.state != KVX_CONN_IN_FLIGHT) return;
    for (const ConnRank &q : r.ranks)
        if (q.expected < 0 || q.done < q.expected) return;
    r.state = r.writes_failed ? KVX_CONN_FAILED : KVX_CONN_DONE;
    emit(k, id, r);
}

// The live record (id, attempt) while IN_FLIGHT, for the producer-side calls. *stale is set when the
// call names an older attempt, which the caller then ignores.
kvx_status in_flight(kvx_conn_s *k, int64_t id, int32_t attempt, int32_t rank, ConnRecord **out, bool *stale) {
    *out = nullptr;
    *stale = false;
    auto it = k->recs.find(id);
    if (it == k->recs.end()) return fail(KVX_EINVAL, "unknown request %lld", (long long)id);
    ConnRecord &r = it->second;
    if (attempt < r.attempt) {
        *stale = true;
        return KVX_OK;
    }
    if (attempt > r.attempt)
        return fail(KVX_EINVAL, "request %lld: attempt %d was never started", (long long)id, attempt);
    if (rank < 0 || rank >= k->cfg.n_ranks) return fail(KVX_EINVAL, "rank %d outside [0, %d)", rank, k->cfg.n_ranks);
    if (r.state != KVX_CONN_IN_FLIGHT)
        return fail(KVX_EINVAL, "request %lld is not in flight (state %d)", (long long)id, r.state);
    *out = &r;
    return KVX_OK;
}

}  // namespace

extern "C" {

kvx_status kvx_conn_create(const kvx_conn_config *cfg, kvx_conn_t *out) {
    if (!out) return fail(KVX_EINVAL, "out is NULL");
    *out = nullptr;
    kvx_conn_config c = {60 * kSecond, 30 * kSecond, 120 * kSecond, 1, 0};
    if (cfg) {
        if (cfg->reserved) return fail(KVX_EINVAL, "kvx_conn_config.reserved must be 0");
        if (cfg->defer_timeout_us < 0 || cfg->transfer_timeout_us < 0 || cfg->recv_abort_timeout_us < 0 ||
            cfg->n_ranks < 0 || cfg->n_ranks > kMaxRanks)
            return fail(KVX_EINVAL, "timeouts must be >= 0 and n_ranks in [0, %d]", kMaxRanks);
        if (cfg->defer_timeout_us) c.defer_timeout_us = cfg->defer_timeout_us;
        if (cfg->transfer_timeout_us) c.transfer_timeout_us = cfg->transfer_timeout_us;
        if (cfg->recv_abort_timeout_us) c.recv_abort_timeout_us = cfg->recv_abort_timeout_us;
        if (cfg->n_ranks) c.n_ranks = cfg->n_ranks;
    }
    kvx_conn_s *k = new (std::nothrow) kvx_conn_s();
    if (!k) return fail(KVX_ENOMEM, "host allocation failed");
    k->cfg = c;
    *out = k;
    return KVX_OK;
}

kvx_status kvx_conn_destroy(kvx_conn_t k) {
    delete k;
    return KVX_OK;
}

kvx_status kvx_conn_register(kvx_conn_t k, int64_t id, int32_t attempt, const int32_t *dst_ids, int32_t n_dst,
                             int64_t now_us) {
    if (!k || attempt < 0 || n_dst < 0 || (n_dst > 0 && !dst_ids)) return fail(KVX_EINVAL, "bad arguments");
    std::lock_guard<std::mutex> lk(k->mu);
    ConnRecord *r = record_for(k, id, attempt);
    if (!r) return KVX_OK;                                            // stale registration
    if (r->registered) {                                              // resent registration
        if ((int32_t)r->dst.size() != n_dst || !std::equal(r->dst.begin(), r->dst.end(), dst_ids))
            return fail(KVX_EINVAL, "request %lld attempt %d registered twice with different blocks",
                        (long long)id, attempt);
        return KVX_OK;
    }
    if (r->state == KVX_CONN_EXPIRED)
        return fail(KVX_ETIMEDOUT, "request %lld attempt %d: the producer gave up after defer_timeout",
                    (long long)id, attempt);
    r->dst.assign(dst_ids, dst_ids + n_dst);
    r->registered = true;
    add_deadline(k, now_us + k->cfg.recv_abort_timeout_us, id, *r, kAbort);
    rendezvous(k, id, *r, now_us);
    return KVX_OK;
}

kvx_status kvx_conn_prefill(kvx_conn_t k, int64_t id, int32_t attempt, const int32_t *src_ids, int32_t n_src,
                            int64_t n_tokens, int32_t last_chunk, int64_t now_us) {
    if (!k || attempt < 0 || n_src < 0 || n_tokens < 0 || (n_src > 0 && !src_ids))
        return fail(KVX_EINVAL, "bad arguments");
    std::lock_guard<std::mutex> lk(k->mu);
    ConnRecord *r = record_for(k, id, attempt);
    if (!r) return KVX_OK;                                            // a chunk of an older attempt
    if (r->prefill_done || terminal(r->state))
        return fail(KVX_EINVAL, "request %lld attempt %d: a prefill chunk after the last one", (long long)id, attempt);
    r->src.insert(r->src.end(), src_ids, src_ids + n_src);           // chunks collect until the last
    r->n_tokens = n_tokens;
    r->n_chunks += 1;
    if (last_chunk) {
        r->prefill_done = true;
        rendezvous(k, id, *r, now_us);
    }
    return KVX_OK;
}

kvx_status kvx_conn_poll(kvx_conn_t k, int64_t now_us, kvx_conn_event *out, int32_t cap, int32_t *n) {
    if (!k || !n || cap < 0 || (cap > 0 && !out)) return fail(KVX_EINVAL, "bad arguments");
    std::lock_guard<std::mutex> lk(k->mu);
    while (!k->deadlines.empty() && k->deadlines.begin()->first <= now_us) {
        const Deadline d = k->deadlines.begin()->second;
        k->deadlines.erase(k->deadlines.begin());
        auto it = k->recs.find(d.req_id);
        if (it == k->recs.end() || it->second.serial != d.serial) continue;   // released or restarted
        ConnRecord &r = it->second;
        int32_t to = -1;
        if (d.kind == kDefer && r.state == KVX_CONN_DEFERRED) to = KVX_CONN_EXPIRED;
        if (d.kind == kTransfer && r.state == KVX_CONN_IN_FLIGHT) to = KVX_CONN_TIMED_OUT;
        if (d.kind == kAbort && !terminal(r.state)) to = KVX_CONN_ABORTED;
        if (to < 0) continue;
        r.state = to;
        emit(k, d.req_id, r);
    }
    int32_t m = 0;
    while (m < cap && !k->events.empty()) {
        const ConnEvent e = k->events.front();
        k->events.pop_front();
        auto it = k->recs.find(e.req_id);
        if (it == k->recs.end() || it->second.serial != e.serial) continue;
        out[m++] = kvx_conn_event{e.req_id, e.attempt, e.state};
    }
    *n = m;
    return KVX_OK;
}

kvx_status kvx_conn_get(kvx_conn_t k, int64_t id, kvx_conn_info *out) {
    if (!k || !out) return fail(KVX_EINVAL, "bad arguments");
    std::lock_guard<std::mutex> lk(k->mu);
    auto it = k->recs.find(id);
    if (it == k->recs.end()) return fail(KVX_EINVAL, "unknown request %lld", (long long)id);
    const ConnRecord &r = it->second;
    kvx_conn_info f{};
    f.attempt = r.attempt;
    f.state = r.state;
    f.n_tokens = r.n_tokens;
    f.n_src = (int32_t)r.src.size();
    f.n_dst = (int32_t)r.dst.size();
    f.n_chunks = r.n_chunks;
    for (const ConnRank &q : r.ranks) {
        f.writes_issued += q.issued;
        f.writes_done += q.done;
        if (q.expected >= 0) {
            f.ranks_sealed += 1;
            f.writes_expected += q.expected;
        }
    }
    f.writes_failed = r.writes_failed;
    f.n_load_errors = (int32_t)r.load_errors.size();
    f.first_error = -1;
    for (int32_t p = 0; p < (int32_t)r.dst.size() && f.first_error < 0; ++p)
        if (std::find(r.load_errors.begin(), r.load_errors.end(), r.dst[p]) != r.load_errors.end()) f.first_error = p;
    *out = f;
    return KVX_OK;
}

kvx_status kvx_conn_ids(kvx_conn_t k, int64_t id, int32_t *src, int32_t src_cap, int32_t *dst, int32_t dst_cap) {
    if (!k || src_cap < 0 || dst_cap < 0 || (src_cap > 0 && !src) || (dst_cap > 0 && !dst))
        return fail(KVX_EINVAL, "bad arguments");
    std::lock_guard<std::mutex> lk(k->mu);
    auto it = k->recs.find(id);
    if (it == k->recs.end()) return fail(KVX_EINVAL, "unknown request %lld", (long long)id);
    const ConnRecord &r = it->second;
    if ((int64_t)r.src.size() > src_cap || (int64_t)r.dst.size() > dst_cap)
        return fail(KVX_ERANGE, "id arrays need %zu and %zu entries", r.src.size(), r.dst.size());
    std::copy(r.src.begin(), r.src.end(), src);
    std::copy(r.dst.begin(), r.dst.end(), dst);
    return KVX_OK;
}

kvx_status kvx_conn_start(kvx_conn_t k, int64_t id, int32_t attempt, int64_t now_us) {
    if (!k) return fail(KVX_EINVAL, "NULL connector");
    std::lock_guard<std::mutex> lk(k->mu);
    auto it = k->recs.find(id);
    if (it == k->recs.end() || it->second.attempt != attempt)
        return fail(KVX_EINVAL, "request %lld attempt %d unknown", (long long)id, attempt);
    ConnRecord &r = it->second;
    if (r.state != KVX_CONN_READY)
        return fail(KVX_EINVAL, "request %lld is not READY (state %d)", (long long)id, r.state);
    r.state = KVX_CONN_IN_FLIGHT;
    add_deadline(k, now_us + k->cfg.transfer_timeout_us, id, r, kTransfer);
    return KVX_OK;
}

kvx_status kvx_conn_write_issued(kvx_conn_t k, int64_t id, int32_t attempt, int32_t rank, int32_t n_writes) {
    if (!k || n_writes < 0) return fail(KVX_EINVAL, "bad arguments");
    std::lock_guard<std::mutex> lk(k->mu);
    ConnRecord *r;
    bool stale;
    kvx_status st = in_flight(k, id, attempt, rank, &r, &stale);
    if (st != KVX_OK || stale) return st;
    if (r->ranks[rank].expected >= 0)
        return fail(KVX_EINVAL, "request %lld rank %d already sealed", (long long)id, rank);
    r->ranks[rank].issued += n_writes;
    return KVX_OK;
}

kvx_status kvx_conn_seal(kvx_conn_t k, int64_t id, int32_t attempt, int32_t rank) {
    if (!k) return fail(KVX_EINVAL, "NULL connector");
    std::lock_guard<std::mutex> lk(k->mu);
    ConnRecord *r;
    bool stale;
    kvx_status st = in_flight(k, id, attempt, rank, &r, &stale);
    if (st != KVX_OK || stale) return st;
    ConnRank &q = r->ranks[rank];
    if (q.expected < 0) q.expected = q.issued;                        // the writes actually queued
    complete_if_counted(k, id, *r);
    return KVX_OK;
}

kvx_status kvx_conn_write_done(kvx_conn_t k, int64_t id, int32_t attempt, int32_t rank, const int32_t *layer_states,
                               int32_t n_layers, const int32_t *failed_blocks, int32_t n_failed, int64_t now_us) {
    (void)now_us;
    if (!k || n_layers <= 0 || !layer_states || n_failed < 0 || (n_failed > 0 && !failed_blocks))
        return fail(KVX_EINVAL, "bad arguments");
    std::lock_guard<std::mutex> lk(k->mu);
    ConnRecord *r;
    bool stale;
    kvx_status st = in_flight(k, id, attempt, rank, &r, &stale);
    if (st != KVX_OK || stale) return st;
    ConnRank &q = r->ranks[rank];
    if (q.done >= (q.expected >= 0 ? q.expected : q.issued))
        return fail(KVX_EINVAL, "request %lld rank %d: more writes reported than queued", (long long)id, rank);
    // the write's state is decided over all its layers, not the last one reported
    bool failed = false;
    for (int32_t l = 0; l < n_layers; ++l) {
        const int32_t s = layer_states[l];
        if (s == KVX_LAYER_FAILED) failed = true;
        else if (s != KVX_LAYER_DONE)
            return fail(KVX_EINVAL, "request %lld: layer %d of a finished write is %s", (long long)id, l,
                        s == KVX_LAYER_PENDING ? "PENDING" : "not DONE or FAILED");
    }
    q.done += 1;
    if (failed) {
        r->writes_failed += 1;
        const int32_t *b = n_failed ? failed_blocks : r->dst.data();
        const int32_t nb = n_failed ? n_failed : (int32_t)r->dst.size();
        for (int32_t i = 0; i < nb; ++i)
            if (std::find(r->load_errors.begin(), r->load_errors.end(), b[i]) == r->load_errors.end())
                r->load_errors.push_back(b[i]);
    }
    complete_if_counted(k, id, *r);
    return KVX_OK;
}

kvx_status kvx_conn_load_errors(kvx_conn_t k, int64_t id, int32_t *blocks, int32_t cap, int32_t *n) {
    if (!k || !n || cap < 0 || (cap > 0 && !blocks)) return fail(KVX_EINVAL, "bad arguments");
    std::lock_guard<std::mutex> lk(k->mu);
    auto it = k->recs.find(id);
    if (it == k->recs.end()) return fail(KVX_EINVAL, "unknown request %lld", (long long)id);
    const std::vector<int32_t> &e = it->second.load_errors;
    *n = (int32_t)e.size();
    std::copy(e.begin(), e.begin() + std::min<size_t>(e.size(), (size_t)cap), blocks);
    return KVX_OK;
}

kvx_status kvx_conn_release(kvx_conn_t k, int64_t id) {
    if (!k) return fail(KVX_EINVAL, "NULL connector");
    std::lock_guard<std::mutex> lk(k->mu);
    k->recs.erase(id);   // its deadlines and events are dropped when reached (serial no longer found)
    return KVX_OK;
}

int64_t kvx_conn_size(kvx_conn_t k) {
    if (!k) return 0;
    std::lock_guard<std::mutex> lk(k->mu);
    return (int64_t)k->recs.size();
}

}  // extern "C"
