// Host side of the decode plan (lazyattn.h, "decode plan"): grouping a batch's
// pages into runs that several requests read, and the work units and partial
// slots of the document-major decode.
//
// LazyAttention §3 "Problem statement": several requests of one batch read one
// document at different global offsets. With keys stored without position,
// a run of pages is the same data for every request that reads it; only the
// offset differs, and Fact 3.2 (q^T R_{n-m} k depends on n - m) moves that
// offset onto q. So a run is read once per group of its readers.
#include <string.h>

#include <algorithm>
#include <map>
#include <new>
#include <tuple>
#include <vector>

#include "internal.h"

using namespace lazyattn;

namespace {

// Longest run one unit walks (pages): longer runs are cut into pieces of this
// many pages, so that units stay comparable in length (and the kernel's
// producer warp holds a unit's entries two per lane).
constexpr int32_t kMaxUnitPages = 64;

struct Reader {
    int32_t request;
    int32_t entry;    // batch entry of the run's first page in this request's table
};

struct Run {
    int32_t first_page;
    int32_t n_pages;
    std::vector<Reader> readers;
};

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" {

int lazyattn_decode_plan_create(lazyattn_pool_t pool, const uint64_t* E, const int32_t* off,
                                const int32_t* delta, int32_t R, lazyattn_plan_t* out_plan) {
    if (!out_plan) return LAZYATTN_EINVAL;
    *out_plan = nullptr;
    if (!pool || !off || R < 1 || R > 65535) return LAZYATTN_EINVAL;
    if (pool->d.dtype != LAZYATTN_BF16) return LAZYATTN_EDTYPE;
    const bool local = pool->d.key_storage == LAZYATTN_KEYS_DOC_LOCAL;
    if (local && !delta && off[R] > off[0]) return LAZYATTN_EINVAL;
    int32_t bad = -1;
    int rc = lazyattn_check_batch_host(E, off, R, pool->d.num_pages, pool->d.max_position, &bad);
    if (rc != LAZYATTN_OK) return rc;

    lazyattn_plan* plan = new (std::nothrow) lazyattn_plan();
    if (!plan) return LAZYATTN_ENOSPC;
    try {
        const int32_t g = pool->d.n_q_heads / pool->d.n_kv_heads;
        const int32_t users_per_unit = 128 / g;
        plan->num_requests = R;
        plan->g = g;
        plan->hkv = pool->d.n_kv_heads;
        plan->key_storage = pool->d.key_storage;

        // 1. Per request: its trailing writable run (private), and maximal
        // stretches of the other entries with tokens at consecutive page ids
        // and consecutive logical positions (doc-local pools: and a document
        // offset that does not decrease, so a stretch's relative rotations are
        // non-negative).
        struct Stretch {
            int32_t request, entry, n;
        };
        std::vector<Stretch> stretches;
        std::vector<std::pair<int32_t, int32_t>> privates(R, {-1, 0});   // (entry, n)
        int64_t logical_pages = 0;
        for (int32_t r = 0; r < R; ++r) {
            const int32_t e0 = off[r], e1 = off[r + 1];
            int32_t w0 = e1;
            while (w0 > e0 && entry_writable(E[w0 - 1])) --w0;
            if (w0 < e1) {
                privates[r] = {w0, e1 - w0};
                logical_pages += e1 - w0;
            }
            int32_t i = e0;
            while (i < w0) {
                if (entry_nvalid(E[i]) == 0) {
                    ++i;
                    continue;
                }
                int32_t j = i + 1;
                while (j < w0 && entry_nvalid(E[j]) > 0 && entry_page(E[j]) == entry_page(E[j - 1]) + 1 &&
                       entry_start(E[j]) == entry_start(E[j - 1]) + entry_nvalid(E[j - 1]) &&
                       (!local || delta[j] >= delta[j - 1]))
                    ++j;
                stretches.push_back({r, i, j - i});
                logical_pages += j - i;
                i = j;
            }
        }

        // 2. Cut every stretch wherever any stretch starts or ends: the pieces
        // between consecutive cuts are runs that each reader reads whole.
        std::vector<int32_t> cuts;
        cuts.reserve(stretches.size() * 2);
        for (const Stretch& s : stretches) {
            cuts.push_back((int32_t)entry_page(E[s.entry]));
            cuts.push_back((int32_t)entry_page(E[s.entry]) + s.n);
        }
        std::sort(cuts.begin(), cuts.end());
        cuts.erase(std::unique(cuts.begin(), cuts.end()), cuts.end());

        // 3. Pieces with the same pages, token counts, relative positions (and,
        // doc-local, relative document offsets) are one run.
        std::vector<Run> runs;
        std::map<std::vector<int64_t>, int32_t> index;
        std::vector<int64_t> key;
        for (const Stretch& s : stretches) {
            const int32_t p0 = (int32_t)entry_page(E[s.entry]);
            auto it = std::upper_bound(cuts.begin(), cuts.end(), p0);
            int32_t a = p0;
            while (a < p0 + s.n) {
                const int32_t b = std::min<int32_t>(it == cuts.end() ? p0 + s.n : *it, p0 + s.n);
                const int32_t ea = s.entry + (a - p0), n = b - a;
                key.assign({(int64_t)a, (int64_t)n});
                const int32_t st0 = entry_start(E[ea]);
                for (int32_t k = 0; k < n; ++k) {
                    key.push_back(entry_nvalid(E[ea + k]));
                    key.push_back((int64_t)entry_start(E[ea + k]) - st0);
                    if (local) key.push_back((int64_t)delta[ea + k] - delta[ea]);
                }
                auto f = index.find(key);
                int32_t id;
                if (f == index.end()) {
                    id = (int32_t)runs.size();
                    index.emplace(key, id);
                    runs.push_back(Run{a, n, {}});
                } else {
                    id = f->second;
                }
                runs[id].readers.push_back({s.request, ea});
                a = b;
                if (it != cuts.end() && *it == b) ++it;
            }
        }

        // 4. Units: each run in pieces of <= kMaxUnitPages pages, each piece's
        // readers in groups of users_per_unit; longest first, the groups of one
        // piece next to each other (they read the same pages); the private runs
        // last (they wait for the append).
        struct U {
            int32_t n_pages;
            int32_t order;
            PlanUnit unit;
            std::vector<PlanUser> users;
        };
        std::vector<U> units;
        int32_t max_readers = 0;
        int64_t pass_pages = 0;
        auto user_delta = [&](int32_t entry) { return local ? delta[entry] : entry_start(E[entry]); };
        for (const Run& run : runs) {
            max_readers = std::max<int32_t>(max_readers, (int32_t)run.readers.size());
            for (int32_t k0 = 0; k0 < run.n_pages; k0 += kMaxUnitPages) {
                const int32_t n = std::min(kMaxUnitPages, run.n_pages - k0);
                for (size_t u0 = 0; u0 < run.readers.size(); u0 += users_per_unit) {
                    U u;
                    u.n_pages = n;
                    u.order = (int32_t)units.size();
                    u.unit = PlanUnit{run.readers[u0].entry + k0, n, 0, 0};
                    for (size_t k = u0; k < std::min(run.readers.size(), u0 + users_per_unit); ++k) {
                        const Reader& rd = run.readers[k];
                        // the piece's run-local position 0 is the start of its first
                        // entry (position-free) or that entry's document offset
                        // (doc-local), as this request places it
                        u.users.push_back(PlanUser{rd.request, user_delta(rd.entry + k0), 0, 0});
                    }
                    pass_pages += n;
                    units.push_back(std::move(u));
                }
            }
        }
        std::stable_sort(units.begin(), units.end(), [](const U& a, const U& b) { return a.n_pages > b.n_pages; });
        for (int32_t r = 0; r < R; ++r) {   // tail runs, in pieces of <= kMaxUnitPages too
            if (privates[r].first < 0) continue;
            for (int32_t k0 = 0; k0 < privates[r].second; k0 += kMaxUnitPages) {
                U u;
                u.n_pages = std::min(kMaxUnitPages, privates[r].second - k0);
                u.order = (int32_t)units.size();
                u.unit = PlanUnit{privates[r].first + k0, u.n_pages, 0, kUnitPrivate};
                u.users.push_back(PlanUser{r, user_delta(privates[r].first + k0), 0, 0});
                pass_pages += u.n_pages;
                units.push_back(std::move(u));
            }
        }

        // 5. Partial slots: each request's slots are contiguous (pbase[r] ..).
        std::vector<int32_t> pbase(R + 1, 0), fill(R, 0);
        for (const U& u : units)
            for (const PlanUser& us : u.users) ++pbase[us.request + 1];
        for (int32_t r = 0; r < R; ++r) pbase[r + 1] += pbase[r];
        int32_t nusers = 0;
        for (U& u : units) {
            u.unit.user0 = nusers;
            u.unit.n_users = (int32_t)u.users.size() | (u.unit.n_users & kUnitPrivate);
            for (PlanUser& us : u.users) us.partial = pbase[us.request] + fill[us.request]++;
            nusers += (int32_t)u.users.size();
        }

        plan->num_units = (int32_t)units.size();
        plan->num_users = nusers;
        plan->num_partials = pbase[R];
        plan->units_off = 0;
        plan->users_off = up256(units.size() * sizeof(PlanUnit));
        plan->pbase_off = plan->users_off + up256((size_t)nusers * sizeof(PlanUser));
        plan->image.assign(plan->pbase_off + up256((size_t)(R + 1) * sizeof(int32_t)), 0);
        uint8_t* img = plan->image.data();
        PlanUser* up = reinterpret_cast<PlanUser*>(img + plan->users_off);
        for (size_t i = 0; i < units.size(); ++i) {
            memcpy(img + plan->units_off + i * sizeof(PlanUnit), &units[i].unit, sizeof(PlanUnit));
            for (const PlanUser& us : units[i].users) *up++ = us;
        }
        memcpy(img + plan->pbase_off, pbase.data(), (size_t)(R + 1) * sizeof(int32_t));
        plan->stats.units = plan->num_units;
        plan->stats.runs = (int32_t)runs.size() + (int32_t)std::count_if(privates.begin(), privates.end(),
                                                                         [](const auto& p) { return p.first >= 0; });
        plan->stats.partials = plan->num_partials;
        plan->stats.max_readers = max_readers;
        plan->stats.logical_pages = logical_pages;
        plan->stats.pass_pages = pass_pages;
    } catch (...) {
        delete plan;
        return LAZYATTN_ENOSPC;
    }
    *out_plan = plan;
    return LAZYATTN_OK;
}

size_t lazyattn_decode_plan_device_bytes(lazyattn_plan_t plan) { return plan ? plan->image.size() : 0; }

int lazyattn_decode_plan_upload(lazyattn_plan_t plan, void* buf, size_t bytes, void* stream) {
    if (!plan || !buf || bytes < plan->image.size() || (reinterpret_cast<uintptr_t>(buf) & 255u))
        return LAZYATTN_EINVAL;
    if (cudaMemcpyAsync(buf, plan->image.data(), plan->image.size(), cudaMemcpyHostToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LAZYATTN_ECUDA;
    plan->device = buf;
    return LAZYATTN_OK;
}

int lazyattn_decode_plan_get_stats(lazyattn_plan_t plan, lazyattn_decode_plan_stats* out) {
    if (!plan || !out) return LAZYATTN_EINVAL;
    *out = plan->stats;
    return LAZYATTN_OK;
}

int lazyattn_decode_plan_destroy(lazyattn_plan_t plan) {
    if (!plan) return LAZYATTN_EINVAL;
    delete plan;
    return LAZYATTN_OK;
}

}  // extern "C"
