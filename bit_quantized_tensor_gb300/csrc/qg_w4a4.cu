#include "qg_internal.h"
extern "C" int w4a4_quantize(int64_t, int64_t, const float*, int64_t, const uint16_t*, int64_t,
                             uint8_t*, uint16_t*, uint16_t*, int64_t, void*) {
    return QG_ERR_UNSUPPORTED;
}
extern "C" int w4a4_gemm(int64_t, int64_t, int64_t, const uint8_t*, const uint16_t*, const uint8_t*,
                         const uint16_t*, int64_t, const uint16_t*, const uint16_t*, int64_t,
                         const uint16_t*, uint16_t*, int64_t, void*, size_t, void*) {
    return QG_ERR_UNSUPPORTED;
}
