// Thread-local error text and status helpers shared by the host-side entry points.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <string>

#include "splitkv.h"

namespace splitkv {

// Records a printf-style message for splitkv_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);

// Clears the message at the start of a successful call.
void clear_error();

}  // namespace splitkv
