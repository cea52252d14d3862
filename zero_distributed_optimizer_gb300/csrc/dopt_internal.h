// Internal state shared by the host layout code and the CUDA launchers.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "dopt.h"

// Elements per CUDA tile: 256 threads x 8 elements.  The per-tile index into
// the run table is built on the host with the same constant.
constexpr int64_t kDoptTileElems = 2048;

// Run metadata bits: bit 0 = the run's params take weight decay; bits 8..15
// = the rank (inside its instance) that owns the run.
constexpr int32_t kRunDecays = 1;
constexpr int kRunRankShift = 8;

struct dopt_layout {
    dopt_layout_cfg cfg{};  // instances normalised to >= 1
    int32_t R = 1;          // ranks per instance (D / instances)
    int64_t numel = 0;      // padded buffer length

    std::vector<int64_t> param_start, param_end;
    std::vector<int32_t> param_bucket;
    std::vector<uint8_t> param_decays;
    std::vector<dopt_range> buckets;
    std::vector<dopt_piece> pieces;

    // Kernel tables.  A run is a maximal stretch of owned elements of one
    // bucket with one owner rank and one weight-decay flag; the gaps between
    // runs are padding.  tile_run[t] is the first run ending after tile t's start.
    std::vector<int64_t> run_start, run_end;
    std::vector<int32_t> run_meta;
    std::vector<int32_t> tile_run;
    // bucket_run[k] is the first run of bucket k; bucket_run[n_buckets] is
    // the run count.  Runs never cross a bucket boundary.
    std::vector<int32_t> bucket_run;

    // Device copies (one allocation), valid on `device` once uploaded.
    int device = -1;
    void *d_block = nullptr;
    const int64_t *d_run_start = nullptr;
    const int64_t *d_run_end = nullptr;
    const int32_t *d_run_meta = nullptr;
    const int32_t *d_tile_run = nullptr;
};

namespace dopt {

// Record an error message for dopt_last_error and return `code`.
int fail(int code, const char *fmt, ...);
void clear_error();

}  // namespace dopt
