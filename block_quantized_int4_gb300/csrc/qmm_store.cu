// qmm_store.cu -- expert hot-store: a least-recently-used set of experts
// resident in device memory, filled from host memory with asynchronous
// copies, after the Colibri page ("Arquitectura del Sistema": a per-layer LRU
// cache of experts, an optional hot store in RAM or VRAM, and a prefetcher
// that asks for the next layer's experts ahead of use).  Here host memory
// holds every expert (it stands in for the page's disk and page cache) and
// the device keeps n_slots of them; the MoE kernels read the slot arena
// through expert ids remapped to slot ids.
//
// Stream discipline (correct by construction, no host waits):
//  - a slot is overwritten only after the compute stream has passed the
//    release point of every request that used it (the copy stream waits on
//    that release event);
//  - the compute stream waits on the copy stream's last event before any
//    request whose experts were copied since its previous wait, and the slot
//    table on the device is updated on the compute stream after that wait.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>
#include <vector>

#include "qmm.h"
#include "qmm_device.cuh"
#include "qmm_internal.h"

// ---------------------------------------------------------------------------
// Host LRU over integer keys and slots
// ---------------------------------------------------------------------------
struct qmm_lru {
    int32_t n_keys = 0, n_slots = 0;
    std::vector<int32_t> slot_of;     // key -> slot or -1
    std::vector<int32_t> key_of;      // slot -> key or -1
    std::vector<int32_t> prev, next;  // recency list over occupied slots: head = most recent
    int32_t head = -1, tail = -1;
    std::vector<int32_t> free_slots;  // never used yet, taken from the back
    std::vector<uint32_t> use_mark;   // == use_epoch: slot holds a key of the last use request
    std::vector<uint32_t> pf_mark;    // == pf_epoch: slot loaded or refreshed by the running prefetch
    uint32_t use_epoch = 0, pf_epoch = 0;
    int64_t hits = 0, misses = 0, evictions = 0, prefetched = 0;

    void unlink(int32_t s) {
        if (prev[s] >= 0) next[prev[s]] = next[s]; else head = next[s];
        if (next[s] >= 0) prev[next[s]] = prev[s]; else tail = prev[s];
        prev[s] = next[s] = -1;
    }
    void push_front(int32_t s) {
        prev[s] = -1;
        next[s] = head;
        if (head >= 0) prev[head] = s;
        head = s;
        if (tail < 0) tail = s;
    }
    static void bump(uint32_t& epoch, std::vector<uint32_t>& marks) {
        if (++epoch == 0) {  // wrapped: clear the marks
            std::fill(marks.begin(), marks.end(), 0u);
            epoch = 1;
        }
    }
};

namespace {

// The slot for a key that is not resident: a never-used slot, else the least
// recently used slot that holds no key of the last use request and (while
// prefetching) no key this prefetch loaded or refreshed.  -1 if none.
int32_t lru_victim(qmm_lru* c, bool prefetch) {
    if (!c->free_slots.empty()) {
        const int32_t s = c->free_slots.back();
        c->free_slots.pop_back();
        return s;
    }
    for (int32_t s = c->tail; s >= 0; s = c->prev[s])
        if (c->use_mark[s] != c->use_epoch && !(prefetch && c->pf_mark[s] == c->pf_epoch)) return s;
    return -1;
}

// One request over keys[0..n).
//  use != 0: the keys are needed now.  The request's distinct keys must fit
//    in the slots (else QMM_ERR_SHAPE and nothing changes); each distinct key
//    counts once as a hit or a miss; every key of the request is protected
//    from eviction until the next use request; keys become most recent in
//    request order.
//  use == 0: prefetch.  Absent keys are loaded as most recent into slots that
//    hold no key of the last use request; keys that find no such slot are
//    skipped (slot -1).  Resident keys become most recent.
// For each load: load_keys/load_slots (in order) and the key it evicted
// (evicted_keys, -1 for a never-used slot).
qmm_status lru_apply(qmm_lru* c, const int32_t* keys, int32_t n, int use, int32_t* slots_out, int32_t* load_keys,
                     int32_t* load_slots, int32_t* n_loads, int32_t* evicted_keys) {
    for (int32_t i = 0; i < n; ++i)
        if (keys[i] < 0 || keys[i] >= c->n_keys) return QMM_ERR_ARG;
    if (use) {
        std::vector<int32_t> distinct(keys, keys + n);
        std::sort(distinct.begin(), distinct.end());
        if (std::unique(distinct.begin(), distinct.end()) - distinct.begin() > c->n_slots) return QMM_ERR_SHAPE;
        qmm_lru::bump(c->use_epoch, c->use_mark);
    } else {
        qmm_lru::bump(c->pf_epoch, c->pf_mark);
    }
    // pass 1: protect every resident key of the request before any load can
    // pick a victim (a hit counts once per distinct key)
    for (int32_t i = 0; i < n; ++i) {
        const int32_t s = c->slot_of[keys[i]];
        if (s < 0) continue;
        if (use) {
            if (c->use_mark[s] != c->use_epoch) c->hits++;
            c->use_mark[s] = c->use_epoch;
        } else {
            c->pf_mark[s] = c->pf_epoch;
        }
    }
    // pass 2, in request order: resident keys become most recent, absent
    // keys are loaded
    int32_t nl = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t k = keys[i];
        int32_t s = c->slot_of[k];
        if (s >= 0) {
            c->unlink(s);
            c->push_front(s);
        } else {
            s = lru_victim(c, !use);
            if (s < 0) {  // only a prefetch can run out of slots
                if (slots_out) slots_out[i] = -1;
                continue;
            }
            const int32_t old = c->key_of[s];
            if (old >= 0) {
                c->slot_of[old] = -1;
                c->evictions++;
                c->unlink(s);
            }
            if (evicted_keys) evicted_keys[nl] = old;
            c->key_of[s] = k;
            c->slot_of[k] = s;
            c->push_front(s);
            if (use) {
                c->misses++;
                c->use_mark[s] = c->use_epoch;
            } else {
                c->prefetched++;
                c->pf_mark[s] = c->pf_epoch;
            }
            if (load_keys) load_keys[nl] = k;
            if (load_slots) load_slots[nl] = s;
            ++nl;
        }
        if (slots_out) slots_out[i] = s;
    }
    if (n_loads) *n_loads = nl;
    return QMM_OK;
}

}  // namespace

extern "C" {

qmm_status qmm_lru_create(int32_t n_keys, int32_t n_slots, qmm_lru** out) {
    if (!out || n_keys <= 0 || n_slots <= 0) return QMM_ERR_ARG;
    qmm_lru* c = new (std::nothrow) qmm_lru();
    if (!c) return QMM_ERR_ARG;
    c->n_keys = n_keys;
    c->n_slots = n_slots;
    c->slot_of.assign(n_keys, -1);
    c->key_of.assign(n_slots, -1);
    c->prev.assign(n_slots, -1);
    c->next.assign(n_slots, -1);
    c->use_mark.assign(n_slots, 0u);
    c->pf_mark.assign(n_slots, 0u);
    c->free_slots.resize(n_slots);
    for (int32_t s = 0; s < n_slots; ++s) c->free_slots[s] = n_slots - 1 - s;  // slot 0 first
    *out = c;
    return QMM_OK;
}

void qmm_lru_destroy(qmm_lru* c) { delete c; }

qmm_status qmm_lru_request(qmm_lru* c, const int32_t* keys, int32_t n, int32_t use, int32_t* slots_out,
                           int32_t* load_keys, int32_t* load_slots, int32_t* n_loads) {
    if (!c || n < 0 || (n > 0 && !keys)) return QMM_ERR_ARG;
    return lru_apply(c, keys, n, use, slots_out, load_keys, load_slots, n_loads, nullptr);
}

qmm_status qmm_lru_stats(const qmm_lru* c, int64_t* hits, int64_t* misses, int64_t* evictions, int64_t* prefetched) {
    if (!c) return QMM_ERR_ARG;
    if (hits) *hits = c->hits;
    if (misses) *misses = c->misses;
    if (evictions) *evictions = c->evictions;
    if (prefetched) *prefetched = c->prefetched;
    return QMM_OK;
}

qmm_status qmm_lru_slot_of(const qmm_lru* c, int32_t key, int32_t* slot) {
    if (!c || !slot || key < 0 || key >= c->n_keys) return QMM_ERR_ARG;
    *slot = c->slot_of[key];
    return QMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Device side: slot-table updates and id remapping
// ---------------------------------------------------------------------------
namespace qmm {
namespace {

constexpr int TABLE_UPDATES = 32;  // (key, slot) pairs per update launch

struct TableUpdate {
    int32_t key[TABLE_UPDATES];
    int32_t slot[TABLE_UPDATES];  // -1: the key left the store
    int32_t n;
};

__global__ void store_table_kernel(int32_t* __restrict__ slot_of, TableUpdate u) {
    // evictions first, then loads, so a key evicted and reloaded in one batch ends resident
    if (threadIdx.x == 0)
        for (int i = 0; i < u.n; ++i) slot_of[u.key[i]] = u.slot[i];
}

__global__ void store_map_kernel(const int32_t* __restrict__ ids, int64_t n, const int32_t* __restrict__ slot_of,
                                 int32_t n_keys, int32_t* __restrict__ out, int* err) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t k = ids[i];
        int32_t s = -1;
        if (k >= 0 && k < n_keys) s = slot_of[k];
        if (s < 0) atomicOr(err, ERR_BAD_EXPERT);
        out[i] = s;
    }
}

}  // namespace
}  // namespace qmm

struct qmm_store {
    qmm_lru* lru = nullptr;
    std::vector<qmm_store_plane> planes;
    int32_t* dev_slot_of = nullptr;  // device [E]
    int dev = 0;
    // release events: slot s may be overwritten once rel[slot_rel[s]] has completed
    std::vector<cudaEvent_t> rel;
    std::vector<int> slot_rel;  // -1: never used by a request
    int rel_next = 0;
    std::vector<int32_t> last_slots;  // slots of the last use request
    bool released = true;             // last_slots carry a release event
    cudaEvent_t copied = nullptr;     // last copy batch
    bool copies_pending = false;      // copies issued since the compute stream last waited
    std::vector<std::pair<int32_t, int32_t>> pending_table;  // (key, slot) changes not yet on the device
    int64_t bytes_copied = 0;
};

namespace {

qmm_status flush_table(qmm_store* st, cudaStream_t compute) {
    using namespace qmm;
    size_t i = 0;
    while (i < st->pending_table.size()) {
        TableUpdate u = {};
        u.n = 0;
        for (; i < st->pending_table.size() && u.n < TABLE_UPDATES; ++i, ++u.n) {
            u.key[u.n] = st->pending_table[i].first;
            u.slot[u.n] = st->pending_table[i].second;
        }
        store_table_kernel<<<1, 32, 0, compute>>>(st->dev_slot_of, u);
        if (cudaGetLastError() != cudaSuccess) return QMM_ERR_CUDA;
    }
    st->pending_table.clear();
    return QMM_OK;
}

// Issue the copies of a planned batch on the copy stream.
qmm_status issue_loads(qmm_store* st, const int32_t* keys, const int32_t* slots, const int32_t* evicted, int32_t nl,
                       cudaStream_t copy) {
    for (int32_t i = 0; i < nl; ++i) {
        const int32_t s = slots[i];
        if (st->slot_rel[s] >= 0 && cudaStreamWaitEvent(copy, st->rel[st->slot_rel[s]], 0) != cudaSuccess)
            return QMM_ERR_CUDA;
        for (const qmm_store_plane& p : st->planes) {
            const char* src = static_cast<const char*>(p.host) + (size_t)keys[i] * (size_t)p.host_stride;
            char* dst = static_cast<char*>(p.dev) + (size_t)s * (size_t)p.bytes;
            if (cudaMemcpyAsync(dst, src, (size_t)p.bytes, cudaMemcpyHostToDevice, copy) != cudaSuccess)
                return QMM_ERR_CUDA;
            st->bytes_copied += p.bytes;
        }
        if (evicted[i] >= 0) st->pending_table.emplace_back(evicted[i], -1);
        st->pending_table.emplace_back(keys[i], s);
    }
    if (nl > 0) {
        if (cudaEventRecord(st->copied, copy) != cudaSuccess) return QMM_ERR_CUDA;
        st->copies_pending = true;
    }
    return QMM_OK;
}

}  // namespace

extern "C" {

qmm_status qmm_store_create(int32_t E, int32_t n_slots, const qmm_store_plane* planes, int32_t n_planes,
                            int32_t* dev_slot_of, qmm_store** out) {
    if (!out || E <= 0 || n_slots <= 0 || n_slots > E || !planes || n_planes <= 0 || n_planes > QMM_STORE_MAX_PLANES ||
        !dev_slot_of)
        return QMM_ERR_ARG;
    for (int32_t p = 0; p < n_planes; ++p)
        if (!planes[p].host || !planes[p].dev || planes[p].bytes <= 0 || planes[p].host_stride < planes[p].bytes)
            return QMM_ERR_ARG;
    int sms = 0, optin = 0;
    if (!qmm::device_facts(&sms, &optin)) return QMM_ERR_DEVICE;
    qmm_store* st = new (std::nothrow) qmm_store();
    if (!st) return QMM_ERR_ARG;
    if (qmm_lru_create(E, n_slots, &st->lru) != QMM_OK) {
        delete st;
        return QMM_ERR_ARG;
    }
    st->planes.assign(planes, planes + n_planes);
    st->dev_slot_of = dev_slot_of;
    cudaGetDevice(&st->dev);
    st->slot_rel.assign(n_slots, -1);
    st->rel.assign(8, nullptr);
    bool ok = cudaEventCreateWithFlags(&st->copied, cudaEventDisableTiming) == cudaSuccess;
    for (auto& e : st->rel) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    // every key starts absent
    ok = ok && cudaMemset(dev_slot_of, 0xff, sizeof(int32_t) * (size_t)E) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        qmm_store_destroy(st);
        return QMM_ERR_CUDA;
    }
    *out = st;
    return QMM_OK;
}

void qmm_store_destroy(qmm_store* st) {
    if (!st) return;
    if (st->copied) cudaEventDestroy(st->copied);
    for (auto& e : st->rel)
        if (e) cudaEventDestroy(e);
    qmm_lru_destroy(st->lru);
    delete st;
}

qmm_status qmm_store_request(qmm_store* st, const int32_t* ids, int32_t n, void* compute_stream, void* copy_stream) {
    if (!st || n < 0 || (n > 0 && !ids)) return QMM_ERR_ARG;
    if (!st->released) {  // the caller did not release the previous request: release it here
        const qmm_status r = qmm_store_release(st, compute_stream);
        if (r != QMM_OK) return r;
    }
    std::vector<int32_t> slots(n), lk(n), ls(n), ev(n);
    int32_t nl = 0;
    qmm_status s = lru_apply(st->lru, ids, n, 1, slots.data(), lk.data(), ls.data(), &nl, ev.data());
    if (s != QMM_OK) return s;
    cudaStream_t compute = static_cast<cudaStream_t>(compute_stream), copy = static_cast<cudaStream_t>(copy_stream);
    s = issue_loads(st, lk.data(), ls.data(), ev.data(), nl, copy);
    if (s != QMM_OK) return s;
    if (st->copies_pending) {
        if (cudaStreamWaitEvent(compute, st->copied, 0) != cudaSuccess) return QMM_ERR_CUDA;
        st->copies_pending = false;
    }
    st->last_slots.assign(slots.begin(), slots.end());
    st->released = false;
    return flush_table(st, compute);
}

qmm_status qmm_store_release(qmm_store* st, void* compute_stream) {
    if (!st) return QMM_ERR_ARG;
    const int r = st->rel_next;
    st->rel_next = (st->rel_next + 1) % (int)st->rel.size();
    if (cudaEventRecord(st->rel[r], static_cast<cudaStream_t>(compute_stream)) != cudaSuccess) return QMM_ERR_CUDA;
    for (int32_t s : st->last_slots) st->slot_rel[s] = r;
    st->released = true;
    return QMM_OK;
}

qmm_status qmm_store_prefetch(qmm_store* st, const int32_t* ids, int32_t n, void* copy_stream) {
    if (!st || n < 0 || (n > 0 && !ids)) return QMM_ERR_ARG;
    std::vector<int32_t> slots(n), lk(n), ls(n), ev(n);
    int32_t nl = 0;
    qmm_status s = lru_apply(st->lru, ids, n, 0, slots.data(), lk.data(), ls.data(), &nl, ev.data());
    if (s != QMM_OK) return s;
    return issue_loads(st, lk.data(), ls.data(), ev.data(), nl, static_cast<cudaStream_t>(copy_stream));
}

qmm_status qmm_store_map_ids(qmm_store* st, const int32_t* ids, int64_t n, int32_t* slot_ids, void* stream) {
    if (!st || n < 0 || (n > 0 && (!ids || !slot_ids))) return QMM_ERR_ARG;
    if (n == 0) return QMM_OK;
    int sms = 0, optin = 0;
    if (!qmm::device_facts(&sms, &optin)) return QMM_ERR_DEVICE;
    const int grid = (int)std::min<int64_t>((n + 255) / 256, 4 * (int64_t)sms);
    qmm::store_map_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        ids, n, st->dev_slot_of, st->lru->n_keys, slot_ids, qmm::device_error_word());
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

qmm_status qmm_store_stats(const qmm_store* st, int64_t* hits, int64_t* misses, int64_t* evictions,
                           int64_t* prefetched, int64_t* bytes_copied) {
    if (!st) return QMM_ERR_ARG;
    qmm_lru_stats(st->lru, hits, misses, evictions, prefetched);
    if (bytes_copied) *bytes_copied = st->bytes_copied;
    return QMM_OK;
}

}  // extern "C"
