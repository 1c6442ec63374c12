// idx_internal.h -- host-side helpers shared by the library's translation
// units (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/idx.h"
#include <nvtx3/nvToolsExt.h>

namespace idx {

// Device address of the sticky status word of the current device.
unsigned int *device_status_ptr();

// Number of SMs of the current device (cached per device).
int sm_count();

// 16-byte alignment check of a device pointer.
inline bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Encode a tiled TMA descriptor of uint8 elements (rank 2 or 3).  Returns
// false if the driver rejects the arguments.
bool encode_tma_u8(CUtensorMap *map, int rank, const void *base, const uint64_t *dims,
                   const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swz);

// Chunked top-k pieces (idx_select.cu) for a logits call that computes the
// top-k's digit-1 histograms itself: the plan kernel (with zero_cvalid it
// also clears the per-chunk valid counts), the phases (hist_done: start at
// the filter), where the counts live in ws, and whether idx_topk would take
// the chunked path for these arguments.
idx_status topk_chunked_plan(const int32_t *lengths, int64_t ld, int rows, void *ws,
                             int zero_cvalid, cudaStream_t s);
idx_status topk_chunked_phases(const float *logits, int64_t ld, int rows, const int32_t *lengths,
                               int k, int32_t *out, int64_t ld_out, void *ws, int vec_ok,
                               int hist_done, cudaStream_t s);
int topk_chunked_counts(void *ws, int rows, int64_t ld, uint32_t **hist, uint32_t **valid,
                        uint32_t **cvalid);
bool topk_takes_chunked(const float *logits, int64_t ld, int rows, int k, const void *ws,
                        size_t ws_bytes);

// An NVTX range around one C-ABI call, named after the entry point, so a
// profiler's timeline shows which call launched which kernels.  NVTX is
// header-only: without a profiler attached a range costs a test of one
// function pointer.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define IDX_NVTX_RANGE(name) ::idx::NvtxRange idx_nvtx_range_(name)

inline idx_status launch_status(cudaError_t e)
{
    return e == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel on the stream finishes; it must call pdl_wait() before
// touching memory an earlier kernel may use.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

} // namespace idx
