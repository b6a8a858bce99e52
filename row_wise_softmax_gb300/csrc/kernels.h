// Internal interface between the C ABI (softmax_abi.cu), the scheduler
// (plan.cpp) and the kernel translation units.  Not installed; the public
// interface is include/softmax.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "softmax.h"

namespace rwsm {

struct Problem {
    const void* in;
    void* out;
    int64_t n_rows, n_cols, ld_in, ld_out;
    int dtype;
    bool no_bulk = false;   // rows live in host memory: no cp.async.bulk staging
};

// Scheduler (plan.cpp): validation and the path / launch-shape decision.
int validate(const void* in, const void* out, int64_t n_rows, int64_t n_cols,
             int64_t ld_in, int64_t ld_out, int dtype);
int make_plan(const softmax_device_desc_t& dev, const Problem& p, int path,
              softmax_plan_t* plan);
// Is a caller-supplied plan safe and complete for this problem?
int check_plan(const softmax_device_desc_t& dev, const Problem& p, const softmax_plan_t& plan);

// Launchers, one per path (each in its own translation unit).
cudaError_t launch_warp_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_tile_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_row_slices(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_twopass(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_stream_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);

// Largest cluster the row-slice kernel can launch with on the current device.
int max_cluster_size_row_slices();

// Error words of the translation units that wait on mbarriers: read and
// optionally clear (host side, after the device has been synchronised).
unsigned read_error_row_slices(bool clear);
unsigned read_error_tile_rows(bool clear);
unsigned read_error_stream_rows(bool clear);
cudaError_t launch_selftest_wait(cudaStream_t s);

// Launch attributes shared by every kernel launch: a cluster dimension when
// cs > 1, and programmatic stream serialisation (the kernels begin with
// griddepcontrol.wait).  Returns the number of attributes written (<= 2).
inline int launch_attrs(cudaLaunchAttribute* a, int cs)
{
    int n = 0;
    if (cs > 1) {
        a[n].id = cudaLaunchAttributeClusterDimension;
        a[n].val.clusterDim.x = static_cast<unsigned>(cs);
        a[n].val.clusterDim.y = 1;
        a[n].val.clusterDim.z = 1;
        ++n;
    }
    a[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    return n;
}

// Persistent grid size for `work` equal units (rows, tiles, row groups)
// dealt round-robin to at most `max_active` resident CTAs (or clusters):
// the last round should be as full as possible (the tail effect of the cs336
// lecture 6 notes, "Block Occupancy", applied to units per CTA).  Among
// g in [max_active/2, max_active], take those whose idle share of the last
// round, (g * ceil(work/g) - work) / (g * ceil(work/g)), is within 1% of the
// best; prefer a multiple of `sm_count`, then the largest.
inline int64_t balanced_grid(int64_t work, int64_t max_active, int64_t sm_count)
{
    if (work <= 0 || max_active <= 0)
        return 1;
    if (work <= max_active)
        return work;
    const int64_t lo = (max_active + 1) / 2;
    double best = 1.0;
    for (int64_t g = lo; g <= max_active; ++g) {
        const int64_t slots = g * ((work + g - 1) / g);
        const double idle = static_cast<double>(slots - work) / static_cast<double>(slots);
        if (idle < best)
            best = idle;
    }
    int64_t pick = -1, pick_mult = -1;
    for (int64_t g = lo; g <= max_active; ++g) {
        const int64_t slots = g * ((work + g - 1) / g);
        const double idle = static_cast<double>(slots - work) / static_cast<double>(slots);
        if (idle > best + 0.01)
            continue;
        pick = g;
        if (sm_count > 0 && g % sm_count == 0)
            pick_mult = g;
    }
    return pick_mult > 0 ? pick_mult : pick;
}

// Helpers implemented in softmax_abi.cu.
int resident_ctas(const void* kernel, int threads, int smem_bytes);  // whole-GPU CTA slots
int sm_count_current();
void note_launch();

}  // namespace rwsm
