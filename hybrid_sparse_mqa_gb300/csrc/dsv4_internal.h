// dsv4_internal.h - host helpers shared by the library's translation units
// (not part of the C ABI; hidden from the shared library's symbol table).
#ifndef DSV4_INTERNAL_H
#define DSV4_INTERNAL_H

#include "dsv4attn.h"

namespace dsv4 {

// Host-side checks of a pool descriptor: DSV4_OK, DSV4_ERR_INVALID (null
// pointers, no pages, empty page table, rows not 16-byte aligned) or
// DSV4_ERR_UNSUPPORTED (page size other than 256, row size that does not
// match the format).
__attribute__((visibility("hidden"))) int check_pool(const dsv4_kv_pool* pool);

// Device address of the per-device error word that
// dsv4_attn_get_device_error() reads and clears (current device); nullptr if
// the runtime cannot provide it.
__attribute__((visibility("hidden"))) unsigned int* device_error_word();

}  // namespace dsv4

#endif
