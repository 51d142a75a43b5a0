// pkv_decode for MLA (latent attention over a single latent kv head).
#include "pkv_internal.cuh"

namespace pkv {
namespace mla {

pkv_status validate(const pkv_decode_args *a, bool check_ptrs) {
    (void)a;
    (void)check_ptrs;
    return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): not built yet");
}

size_t workspace_size(const pkv_decode_args *a) {
    (void)a;
    return 0;
}

pkv_status launch(const pkv_decode_args *a, void *ws, size_t ws_bytes, int32_t *err, cudaStream_t s) {
    (void)a; (void)ws; (void)ws_bytes; (void)err; (void)s;
    return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): not built yet");
}

}  // namespace mla
}  // namespace pkv
