// fp_sparse_attn_noalloc: the sparse-attention entry point for callers that
// cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: a plugin inside
// a host framework that owns every device allocation and exposes none to its
// plugins, or a serving loop running under a fixed device-memory budget where
// a new allocation could fail mid-request (and cudaMalloc would also stall
// the device while it synchronises).  For them, the scratch that
// fp_sparse_attn keeps in its workspace (status word, work schedule, bf16
// copies of the block means) lives here in one file-scope device array of
// FP_NOALLOC_SCRATCH_BYTES, reserved on every GPU that loads the library for
// as long as the process lives.  The computation is exactly fp_sparse_attn's:
// this file only supplies that array as its workspace.
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"

// The built-in scratch.  In host code this name is only a host-side stand-in
// for the device symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char fp_noalloc_scratch[FP_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array in the caller's current context.  It
// is looked up on every call and never cached: an address belongs to the
// context it came from, and a caller may make a non-primary context current,
// or reset the device (which destroys the context), between calls.  The
// lookup is a host-side table read once the module is loaded; the first call
// in a context may load it, which is why that call must come before any
// stream capture.
fp_status scratch_in_current_context(void **addr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, fp_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        const char *dbg = getenv("FPREFILL_DEBUG");
        if (dbg && *dbg && *dbg != '0') fprintf(stderr, "[fprefill] scratch address: %s\n", cudaGetErrorString(e));
        return FP_ERR_CUDA;
    }
    *addr = p;
    return FP_OK;
}

}  // namespace

extern "C" fp_status fp_sparse_attn_noalloc(const fp_problem *p, const fp_params *prm, const int *row_ptr,
                                            const int *col_idx, const float *k_mean, const float *v_mean,
                                            void *out, float *lse_opt, int *status_dev_opt, void *stream) {
    // The fixed scratch does not split rows unless the caller asks for it
    // (kv_splits 0 means 1 here): split-KV partial outputs would crowd it.
    fp_params q;
    if (prm) {
        q = *prm;
        if (q.kv_splits == 0) q.kv_splits = 1;
        prm = &q;
    }
    // Argument checks first, with no workspace: every argument error comes back
    // as from fp_sparse_attn; FP_ERR_WORKSPACE means the arguments are fine.
    fp_status s = fp_sparse_attn(p, prm, row_ptr, col_idx, k_mean, v_mean, out, lse_opt, nullptr, 0, stream);
    if (s != FP_ERR_WORKSPACE) return s == FP_OK ? FP_ERR_INVALID : s;
    const size_t need = fp_attn_workspace_size(p, prm);
    if (need == 0 || need > FP_NOALLOC_SCRATCH_BYTES) {
        const char *dbg = getenv("FPREFILL_DEBUG");
        if (dbg && *dbg && *dbg != '0')
            fprintf(stderr, "[fprefill] no-alloc attention needs %zu bytes of scratch, built-in limit %zu\n", need,
                    (size_t)FP_NOALLOC_SCRATCH_BYTES);
        return FP_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    if ((s = scratch_in_current_context(&scratch)) != FP_OK) return s;
    // the array keeps the previous call's contents: the status word must start at zero
    if ((s = fp_reset_status(scratch, stream)) != FP_OK) return s;
    s = fp_sparse_attn(p, prm, row_ptr, col_idx, k_mean, v_mean, out, lse_opt, scratch, FP_NOALLOC_SCRATCH_BYTES,
                       stream);
    if (s == FP_OK && status_dev_opt &&
        cudaMemcpyAsync(status_dev_opt, scratch, sizeof(int), cudaMemcpyDeviceToDevice, (cudaStream_t)stream) !=
            cudaSuccess)
        return FP_ERR_CUDA;
    return s;
}
