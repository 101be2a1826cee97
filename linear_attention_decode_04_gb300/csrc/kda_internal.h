// kda_internal.h -- helpers shared by the translation units of the library
// (not part of the C ABI; hidden from the exported symbol table).
#pragma once

#define KDA_INTERNAL __attribute__((visibility("hidden")))

// Record a message for kda_last_error() and return `code`.
KDA_INTERNAL int kda_internal_fail(int code, const char* fmt, ...);
// Clear the message of kda_last_error() at the start of a call.
KDA_INTERNAL void kda_internal_clear_error();
