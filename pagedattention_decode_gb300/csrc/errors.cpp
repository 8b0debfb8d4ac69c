// errors.cpp -- status strings and the thread-local last-error message.
#include "internal.h"

namespace pkv {

static thread_local std::string g_last_error;

pkv_status fail(pkv_status status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = std::string(pkv_status_string(status)) + ": " + buf;
    return status;
}

pkv_status ok() {
    g_last_error.clear();
    return PKV_OK;
}

}  // namespace pkv

extern "C" {

int32_t pkv_abi_version(void) { return 1; }

const char *pkv_last_error(void) { return pkv::g_last_error.c_str(); }

const char *pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_DTYPE: return "PKV_ERR_DTYPE";
        case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE";
        case PKV_ERR_OUT_OF_RANGE: return "PKV_ERR_OUT_OF_RANGE";
        case PKV_ERR_EXHAUSTED: return "PKV_ERR_EXHAUSTED";
        case PKV_ERR_DOUBLE_FREE: return "PKV_ERR_DOUBLE_FREE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        default: return "PKV_ERR_UNKNOWN";
    }
}

}  // extern "C"
