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

extern "C" int32_t gs_param_rows(int32_t sh_degree) { return gs::param_rows(sh_degree); }

extern "C" int32_t gs_param_stride(int32_t sh_degree) { return gs::param_stride(sh_degree); }

extern "C" int64_t gs_num_tiles(int32_t width, int32_t height)
{
    if (width <= 0 || height <= 0) return 0;
    return (int64_t)gs::tiles_x_of(width) * gs::tiles_y_of(height);
}

extern "C" const char* gs_version(void) { return "gs-gb300 0.1 sm_103a"; }
