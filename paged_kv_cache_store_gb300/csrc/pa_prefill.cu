// pa_prefill.cu -- varlen causal prefill attention (tcgen05 kernel pending).
#include "pa_internal.cuh"

extern "C" pa_status pa_prefill_varlen(void *, const void *, int64_t, const void *, const void *,
                                       int64_t, const int32_t *, int32_t, const int32_t *,
                                       const int32_t *, int32_t, int32_t, int32_t, int32_t, int32_t,
                                       int32_t, int32_t, int32_t, float, int32_t, pa_stream_t) {
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_prefill_varlen is not built yet");
}
