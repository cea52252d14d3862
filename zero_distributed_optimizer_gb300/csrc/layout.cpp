// Host side of the library: the flat-buffer layout, the four-way range map
// (Megatron-LM distributed-optimizer page, §2, §3, §4.1, §5), the kernel's
// run table, and the device upload of that table.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <new>

#include <cuda_runtime_api.h>

#include "dopt_internal.h"

namespace dopt {

static thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

void clear_error() { g_last_error.clear(); }

namespace {

// Greedy buckets and padding: params at consecutive offsets; the open
// bucket closes once its unpadded count reaches bucket_elems; each bucket
// is padded to a multiple of R * pad_unit (distributed-optimizer page, §2 and §5).
void place_params(dopt_layout &L, const int64_t *sizes, int32_t n) {
    const int64_t unit = int64_t(L.R) * L.cfg.pad_unit;
    L.param_start.resize(n);
    L.param_end.resize(n);
    L.param_bucket.resize(n);
    int64_t cursor = 0;        // next free position in the buffer
    int64_t bucket_begin = 0;  // start of the open bucket
    int32_t first_param = 0;   // first param of the open bucket
    auto close_bucket = [&](int32_t last_param_exclusive) {
        int64_t used = cursor - bucket_begin;
        int64_t padded = ((used + unit - 1) / unit) * unit;
        L.buckets.push_back(dopt_range{bucket_begin, bucket_begin + padded});
        cursor = bucket_begin + padded;
        bucket_begin = cursor;
        first_param = last_param_exclusive;
    };
    for (int32_t p = 0; p < n; ++p) {
        L.param_start[p] = cursor;
        cursor += sizes[p];
        L.param_end[p] = cursor;
        L.param_bucket[p] = int32_t(L.buckets.size());
        if (L.cfg.bucket_elems > 0 && cursor - bucket_begin >= L.cfg.bucket_elems)
            close_bucket(p + 1);
    }
    if (first_param < n) close_bucket(n);
    L.numel = cursor;
}

// Pieces of one bucket by a sweep over the sorted param boundaries and the
// sorted rank boundaries: every step emits the overlap of the current param
// with the current rank's range and advances whichever ends first.
void bucket_pieces(dopt_layout &L, int32_t k, int32_t p_begin, int32_t p_end) {
    const dopt_range b = L.buckets[size_t(k)];
    const int32_t R = L.R;
    const int64_t S = (b.end - b.start) / R;
    if (S == 0) return;
    int32_t p = p_begin, r = 0;
    while (p < p_end && r < R) {
        const int64_t lo = b.start + r * S, hi = lo + S;
        const int64_t a = L.param_start[size_t(p)], e = L.param_end[size_t(p)];
        const int64_t x = std::max(a, lo), y = std::min(e, hi);
        if (x < y) {
            dopt_piece pc{};
            pc.gbuf_world = {x, y};
            pc.gbuf_world_in_bucket = {x - b.start, y - b.start};
            pc.gbuf_local = {x - lo, y - lo};
            pc.param = {x - a, y - a};
            pc.param_id = p;
            pc.bucket_id = k;
            pc.rank = r;
            L.pieces.push_back(pc);
        }
        if (e <= hi)
            ++p;
        else
            ++r;
    }
}

// Runs for the kernel: consecutive pieces of one bucket that touch and
// share the owner rank and the decay flag are merged (the kernel needs
// nothing else per element).  Runs stay inside their bucket, so that a
// launch can cover any contiguous range of buckets.
void build_runs(dopt_layout &L) {
    const int32_t nb = int32_t(L.buckets.size());
    L.bucket_run.assign(size_t(nb) + 1, 0);
    int32_t run_bucket = -1;
    for (const dopt_piece &pc : L.pieces) {
        int32_t meta = (L.param_decays[size_t(pc.param_id)] ? kRunDecays : 0) |
                       (pc.rank << kRunRankShift);
        bool extend = !L.run_end.empty() && L.run_end.back() == pc.gbuf_world.start &&
                      L.run_meta.back() == meta && run_bucket == pc.bucket_id;
        if (extend) {
            L.run_end.back() = pc.gbuf_world.end;
        } else {
            // buckets between the last run's and this one own no run
            for (int32_t k = run_bucket + 1; k <= pc.bucket_id; ++k)
                L.bucket_run[size_t(k)] = int32_t(L.run_start.size());
            run_bucket = pc.bucket_id;
            L.run_start.push_back(pc.gbuf_world.start);
            L.run_end.push_back(pc.gbuf_world.end);
            L.run_meta.push_back(meta);
        }
    }
    for (int32_t k = run_bucket + 1; k <= nb; ++k)
        L.bucket_run[size_t(k)] = int32_t(L.run_start.size());
    const int64_t n_tiles = (L.numel + kDoptTileElems - 1) / kDoptTileElems;
    L.tile_run.resize(size_t(n_tiles) + 1);
    size_t j = 0;
    for (int64_t t = 0; t <= n_tiles; ++t) {
        const int64_t tile_begin = t * kDoptTileElems;
        while (j < L.run_end.size() && L.run_end[j] <= tile_begin) ++j;
        L.tile_run[size_t(t)] = int32_t(j);
    }
}

void release_device(dopt_layout *L) {
    if (L->d_block) {
        int prev = -1;
        cudaGetDevice(&prev);
        if (prev != L->device) cudaSetDevice(L->device);
        cudaFree(L->d_block);
        if (prev >= 0 && prev != L->device) cudaSetDevice(prev);
    }
    L->d_block = nullptr;
    L->d_run_start = L->d_run_end = nullptr;
    L->d_run_meta = L->d_tile_run = nullptr;
    L->device = -1;
}

}  // namespace
}  // namespace dopt

using namespace dopt;

extern "C" {

int dopt_build_range_map(const int64_t *param_sizes, int32_t n_params, const uint8_t *wd_mask,
                         const dopt_layout_cfg *cfg, dopt_layout **out) {
    clear_error();
    if (!out) return fail(DOPT_E_ARG, "dopt_build_range_map: out is NULL");
    *out = nullptr;
    if (!cfg) return fail(DOPT_E_ARG, "dopt_build_range_map: cfg is NULL");
    if (n_params < 0) return fail(DOPT_E_ARG, "dopt_build_range_map: n_params < 0");
    if (n_params > 0 && !param_sizes)
        return fail(DOPT_E_ARG, "dopt_build_range_map: param_sizes is NULL");
    if (cfg->D < 1 || cfg->D > DOPT_MAX_D)
        return fail(DOPT_E_ARG, "dopt_build_range_map: D=%d outside 1..%d", cfg->D, DOPT_MAX_D);
    if (cfg->pad_unit < 1)
        return fail(DOPT_E_ARG, "dopt_build_range_map: pad_unit=%d < 1", cfg->pad_unit);
    if (cfg->bucket_elems < 0)
        return fail(DOPT_E_ARG, "dopt_build_range_map: bucket_elems < 0");
    const int32_t instances = cfg->instances == 0 ? 1 : cfg->instances;
    if (instances < 1 || cfg->D % instances != 0 || cfg->reserved != 0)
        return fail(DOPT_E_ARG, "dopt_build_range_map: instances=%d does not divide D=%d",
                    cfg->instances, cfg->D);
    int64_t total = 0;
    for (int32_t p = 0; p < n_params; ++p) {
        if (param_sizes[p] < 0)
            return fail(DOPT_E_ARG, "dopt_build_range_map: param %d has size %lld < 0", p,
                        (long long)param_sizes[p]);
        total += param_sizes[p];
        if (total > (int64_t(1) << 46))
            return fail(DOPT_E_ARG, "dopt_build_range_map: buffer too large");
    }
    dopt_layout *L = nullptr;
    try {
        L = new dopt_layout();
        L->cfg = *cfg;
        L->cfg.instances = instances;
        L->R = cfg->D / instances;
        L->param_decays.assign(size_t(n_params), 1);
        if (wd_mask)
            for (int32_t p = 0; p < n_params; ++p) L->param_decays[size_t(p)] = wd_mask[p] ? 1 : 0;
        place_params(*L, param_sizes, n_params);
        for (const dopt_range &b : L->buckets)
            if ((b.end - b.start) % L->R != 0) {
                const int32_t R = L->R;
                delete L;
                return fail(DOPT_E_LAYOUT, "bucket [%lld, %lld) does not divide by R=%d",
                            (long long)b.start, (long long)b.end, R);
            }
        if ((L->numel + kDoptTileElems - 1) / kDoptTileElems >= (int64_t(1) << 31)) {
            delete L;
            return fail(DOPT_E_ARG, "dopt_build_range_map: buffer too large");
        }
        int32_t p = 0;
        for (int32_t k = 0; k < int32_t(L->buckets.size()); ++k) {
            int32_t q = p;
            while (q < n_params && L->param_bucket[size_t(q)] == k) ++q;
            bucket_pieces(*L, k, p, q);
            p = q;
        }
        build_runs(*L);
    } catch (const std::bad_alloc &) {
        delete L;
        return fail(DOPT_E_NOMEM, "dopt_build_range_map: out of host memory");
    }
    *out = L;
    return DOPT_OK;
}

int dopt_layout_query(const dopt_layout *L, int64_t *padded_numel, int32_t *n_buckets,
                      int32_t *n_pieces) {
    clear_error();
    if (!L) return fail(DOPT_E_ARG, "dopt_layout_query: layout is NULL");
    if (padded_numel) *padded_numel = L->numel;
    if (n_buckets) *n_buckets = int32_t(L->buckets.size());
    if (n_pieces) *n_pieces = int32_t(L->pieces.size());
    return DOPT_OK;
}

int dopt_layout_buckets(const dopt_layout *L, dopt_range *buckets) {
    clear_error();
    if (!L || (!buckets && !L->buckets.empty()))
        return fail(DOPT_E_ARG, "dopt_layout_buckets: NULL argument");
    std::copy(L->buckets.begin(), L->buckets.end(), buckets);
    return DOPT_OK;
}

int dopt_layout_pieces(const dopt_layout *L, dopt_piece *pieces) {
    clear_error();
    if (!L || (!pieces && !L->pieces.empty()))
        return fail(DOPT_E_ARG, "dopt_layout_pieces: NULL argument");
    std::copy(L->pieces.begin(), L->pieces.end(), pieces);
    return DOPT_OK;
}

int dopt_layout_param_offsets(const dopt_layout *L, dopt_range *params) {
    clear_error();
    if (!L || (!params && !L->param_start.empty()))
        return fail(DOPT_E_ARG, "dopt_layout_param_offsets: NULL argument");
    for (size_t p = 0; p < L->param_start.size(); ++p)
        params[p] = dopt_range{L->param_start[p], L->param_end[p]};
    return DOPT_OK;
}

int dopt_layout_param_ranges(const dopt_layout *L, dopt_range *params) {
    return dopt_layout_param_offsets(L, params);
}

int dopt_layout_to_device(dopt_layout *L) {
    clear_error();
    if (!L) return fail(DOPT_E_ARG, "dopt_layout_to_device: layout is NULL");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(DOPT_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (L->device == dev && (L->d_block || L->run_start.empty())) return DOPT_OK;
    release_device(L);
    const size_t nr = L->run_start.size(), nt = L->tile_run.size();
    const size_t bytes_i64 = nr * sizeof(int64_t);
    const size_t off_end = bytes_i64;
    const size_t off_meta = 2 * bytes_i64;
    const size_t off_tile = off_meta + ((nr * sizeof(int32_t) + 15) / 16) * 16;
    const size_t total = off_tile + nt * sizeof(int32_t);
    if (nr > 0) {
        void *block = nullptr;
        e = cudaMalloc(&block, total);
        if (e != cudaSuccess)
            return fail(DOPT_E_CUDA, "cudaMalloc(%zu): %s", total, cudaGetErrorString(e));
        std::vector<unsigned char> host(total, 0);
        std::copy_n(reinterpret_cast<const unsigned char *>(L->run_start.data()), bytes_i64,
                    host.data());
        std::copy_n(reinterpret_cast<const unsigned char *>(L->run_end.data()), bytes_i64,
                    host.data() + off_end);
        std::copy_n(reinterpret_cast<const unsigned char *>(L->run_meta.data()),
                    nr * sizeof(int32_t), host.data() + off_meta);
        std::copy_n(reinterpret_cast<const unsigned char *>(L->tile_run.data()),
                    nt * sizeof(int32_t), host.data() + off_tile);
        e = cudaMemcpy(block, host.data(), total, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            cudaFree(block);
            return fail(DOPT_E_CUDA, "cudaMemcpy: %s", cudaGetErrorString(e));
        }
        auto *base = static_cast<unsigned char *>(block);
        L->d_block = block;
        L->d_run_start = reinterpret_cast<const int64_t *>(base);
        L->d_run_end = reinterpret_cast<const int64_t *>(base + off_end);
        L->d_run_meta = reinterpret_cast<const int32_t *>(base + off_meta);
        L->d_tile_run = reinterpret_cast<const int32_t *>(base + off_tile);
    }
    L->device = dev;
    return DOPT_OK;
}

void dopt_layout_free(dopt_layout *L) {
    if (!L) return;
    release_device(L);
    delete L;
}

const char *dopt_last_error(void) { return g_last_error.c_str(); }

const char *dopt_version(void) { return "dopt 0.2.0 (sm_103a)"; }

}  // extern "C"
