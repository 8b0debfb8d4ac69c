// internal.h -- library-private helpers shared by the host sources of libpkv.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <string>

#include "pkv.h"

namespace pkv {

// Records a thread-local message for pkv_last_error() and returns `status`.
pkv_status fail(pkv_status status, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
// Clears the thread-local message; returns PKV_OK.
pkv_status ok();

}  // namespace pkv

#define PKV_CHECK_ARG(cond, status, ...)          \
    do {                                          \
        if (!(cond)) return pkv::fail((status), __VA_ARGS__); \
    } while (0)
