// SHA-256 (FIPS 180-4) for prefix-cache block keys.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pa {
void sha256(const void* data, size_t n, uint8_t out[32]);
}
