#include "qg_internal.h"
extern "C" int w4a16_gemm(int64_t, int64_t, int64_t, const uint16_t*, int64_t, const uint8_t*,
                          const uint16_t*, int64_t, uint16_t*, int64_t, void*) {
    return QG_ERR_UNSUPPORTED;
}
