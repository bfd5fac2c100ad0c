// abi.cu -- static helpers of the C ABI (no device work).
#include "gs_common.cuh"

extern "C" const char* gs_error_string(gs_status s)
{
    switch (s) {
        case GS_OK: return "ok";
        case GS_ERR_INVALID_ARG: return "invalid argument";
        case GS_ERR_CAPACITY: return "instance capacity too small";
        case GS_ERR_CUDA: return "CUDA runtime error";
        case GS_ERR_TIMEOUT: return "bounded device wait timed out";
        case GS_ERR_DEVICE: return "device-side error reported";
    }
    return "unknown status";
}

#ifdef GS_CHECKED
namespace gs {
namespace {
constexpr int kMaxReaders = 32;
struct CheckReaders {
    CheckReader f[kMaxReaders];
    int n = 0;
};
// Function-local static: filled by the units' static initializers in whatever
// order the loader runs them.
CheckReaders& check_readers()
{
    static CheckReaders r;
    return r;
}
}  // namespace

void register_check_reader(CheckReader reader)
{
    CheckReaders& r = check_readers();
    if (r.n < kMaxReaders) r.f[r.n++] = reader;
}
}  // namespace gs
#endif

extern "C" gs_status gs_check_report(uint64_t* report, int32_t* checked)
{
    GS_NVTX_RANGE("gs_check_report");
    if (!report || !checked) return GS_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i) report[i] = 0;
#ifdef GS_CHECKED
    *checked = 1;
    GS_CUDA_TRY(cudaDeviceSynchronize());
    const gs::CheckReaders& r = gs::check_readers();
    for (int k = 0; k < r.n; ++k) {
        unsigned long long rec[4];
        GS_CUDA_TRY(r.f[k](rec));
        if (rec[0] != 0 && report[0] == 0) {
            report[1] = rec[1];
            report[2] = rec[2];
            report[3] = rec[3];
        }
        report[0] += rec[0];
    }
    return report[0] ? GS_ERR_DEVICE : GS_OK;
#else
    *checked = 0;
    return GS_OK;
#endif
}

extern "C" int32_t gs_param_rows(int32_t sh_degree) { return gs::param_rows(sh_degree); }

extern "C" int32_t gs_param_stride(int32_t sh_degree) { return gs::param_stride(sh_degree); }

extern "C" int64_t gs_num_tiles(int32_t width, int32_t height)
{
    if (width <= 0 || height <= 0) return 0;
    return (int64_t)gs::tiles_x_of(width) * gs::tiles_y_of(height);
}

extern "C" const char* gs_version(void) { return "gs-gb300 0.1 sm_103a"; }
