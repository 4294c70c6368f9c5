#include "bwd.h"
#include "common.cuh"
namespace attn {
namespace bwd {
size_t workspace_bytes(const Args&) { return 0; }
cudaError_t launch(const Args&, void*, size_t, cudaStream_t, std::string* what) {
    *what = "not built yet";
    return cudaErrorNotSupported;
}
ATTN_DEFINE_STATUS_ACCESSOR(status_exchange)
}  // namespace bwd
}  // namespace attn
