// sfm_noalloc.cu -- sfm_forward() for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain a device buffer at call time: code
// replayed inside a captured CUDA graph whose memory was frozen at capture,
// plug-ins that run under a host framework which owns every allocation, or
// real-time paths where a cudaMalloc (and the implicit synchronisation it may
// bring) is forbidden.  For them the split-KV workspace lives in a fixed
// device array that is part of this library's module: the GPU reserves it when
// the module is loaded and keeps it until the process exits.
//
// Every call on a device uses the same array, so calls whose kernels overlap
// on the GPU (different streams without ordering between them) race on it.
// Nothing in it needs to start at zero: each split writes its partial result
// before the combine kernel of the same call reads it.
#include "sfm_internal.cuh"

namespace {

constexpr size_t kStaticWorkspaceBytes = SFM_NOALLOC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Device address of g_static_workspace on the current device.  In host code
// the symbol itself is only a host-side stand-in, never a device pointer.  The
// address is looked up on every call rather than cached: the lookup allocates
// nothing, and after a device reset (or any re-creation of the primary
// context) the module is loaded again at a new address, which a cached
// pointer would not follow.  The first call on a device loads the module.
int static_workspace(void **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return SFM_ERR_CUDA;
    *out = p;
    return SFM_OK;
}

}  // namespace

extern "C" int sfm_forward_noalloc(const sfm_params *params, const sfm_tensors *inputs, const int32_t *metadata,
                                   size_t metadata_n, float softmax_scale, void *out, float *lse, int32_t *status,
                                   sfm_stream_t stream)
{
    size_t need = 0;
    int rc = sfm_workspace_size(params, &need);
    if (rc) return rc;
    if (need > kStaticWorkspaceBytes) return SFM_ERR_WORKSPACE;
    void *ws = nullptr;
    if (need) {
        rc = static_workspace(&ws);
        if (rc) return rc;
    }
    return sfm_forward(params, inputs, metadata, metadata_n, softmax_scale, out, lse, ws,
                       need ? kStaticWorkspaceBytes : 0, status, stream);
}
