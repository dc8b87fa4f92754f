// trace.cu -- optional kernel-level timing: while enabled, every kernel launch
// of dr_fwd / dr_bwd is bracketed by two CUDA events recorded on the call's
// stream, so a caller can read per-kernel device durations (dr.h, dr_trace_*).
#include <vector>

#include "common.cuh"
#include "trace.cuh"

namespace dr {
namespace {
struct Rec {
    const char* name;
    cudaEvent_t a, b;
};
std::vector<Rec> g_recs;
int g_used = 0;
bool g_on = false;
}  // namespace

TraceScope::TraceScope(const char* name, cudaStream_t st) : st_(st), slot_(-1) {
    if (!g_on || g_used >= (int)g_recs.size()) return;
    slot_ = g_used++;
    g_recs[slot_].name = name;
    cudaEventRecord(g_recs[slot_].a, st_);
}
TraceScope::~TraceScope() {
    if (slot_ >= 0) cudaEventRecord(g_recs[slot_].b, st_);
}

}  // namespace dr

using namespace dr;

extern "C" {

int dr_trace_enable(int max_launches) {
    for (auto& r : g_recs) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_recs.clear();
    g_used = 0;
    g_on = false;
    if (max_launches <= 0) return DR_OK;
    g_recs.resize(max_launches);
    for (auto& r : g_recs) {
        r.name = nullptr;
        if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess)
            return DR_ERR_CUDA;
    }
    g_on = true;
    return DR_OK;
}

int dr_trace_count(void) { return g_used; }

void dr_trace_reset(void) { g_used = 0; }

int dr_trace_get(int i, const char** name, float* ms) {
    if (i < 0 || i >= g_used || !name || !ms) return DR_ERR_INVALID_ARG;
    if (cudaEventSynchronize(g_recs[i].b) != cudaSuccess) return DR_ERR_CUDA;
    if (cudaEventElapsedTime(ms, g_recs[i].a, g_recs[i].b) != cudaSuccess) return DR_ERR_CUDA;
    *name = g_recs[i].name;
    return DR_OK;
}

}  // extern "C"
