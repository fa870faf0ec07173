// SHA-256 as the Secure Hash Standard (FIPS 180-4, section 6.2) defines it: the
// prefix-cache block key of the pages ("KV Cache in Serving Engines", section "4. Prefix
// Caching": the hash defaults to sha256).
//
// The round constants and the initial hash value are not typed in: they are computed
// once from their definition in the standard (the first 32 bits of the fractional
// parts of the cube roots of the first 64 primes, and of the square roots of the first
// 8 primes) with exact integer roots.
#include <stdint.h>
#include <string.h>

#include "pa_sha256.h"

namespace pa {
namespace {

typedef unsigned __int128 u128;

// floor(x^(1/k)) for k = 2 or 3, bit by bit from the top.
uint64_t iroot(u128 x, int k, int bits) {
  uint64_t r = 0;
  for (int b = bits - 1; b >= 0; --b) {
    const uint64_t c = r | (uint64_t(1) << b);
    u128 p = c;
    for (int i = 1; i < k; ++i) p *= c;
    if (p <= x) r = c;
  }
  return r;
}

struct Constants {
  uint32_t k[64];
  uint32_t h0[8];
  Constants() {
    int primes[64], n = 0;
    for (int c = 2; n < 64; ++c) {
      bool prime = true;
      for (int d = 2; d * d <= c; ++d)
        if (c % d == 0) { prime = false; break; }
      if (prime) primes[n++] = c;
    }
    // fractional bits: floor(root(p) * 2^32) mod 2^32 = floor(root(p * 2^(32 k))) mod 2^32
    for (int i = 0; i < 64; ++i) k[i] = (uint32_t)iroot((u128)primes[i] << 96, 3, 40);
    for (int i = 0; i < 8; ++i) h0[i] = (uint32_t)iroot((u128)primes[i] << 64, 2, 40);
  }
};

const Constants& constants() {
  static const Constants c;
  return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void compress(uint32_t h[8], const uint8_t block[64], const uint32_t k[64]) {
  uint32_t w[64];
  for (int t = 0; t < 16; ++t)
    w[t] = (uint32_t)block[4 * t] << 24 | (uint32_t)block[4 * t + 1] << 16 |
           (uint32_t)block[4 * t + 2] << 8 | (uint32_t)block[4 * t + 3];
  for (int t = 16; t < 64; ++t) {
    const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
    const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
    w[t] = s1 + w[t - 7] + s0 + w[t - 16];
  }
  uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
  for (int t = 0; t < 64; ++t) {
    const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    const uint32_t ch = (e & f) ^ (~e & g);
    const uint32_t t1 = hh + S1 + ch + k[t] + w[t];
    const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
    const uint32_t t2 = S0 + maj;
    hh = g;
    g = f;
    f = e;
    e = d + t1;
    d = c;
    c = b;
    b = a;
    a = t1 + t2;
  }
  h[0] += a; h[1] += b; h[2] += c; h[3] += d;
  h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
}

}  // namespace

void sha256(const void* data, size_t n, uint8_t out[32]) {
  const Constants& c = constants();
  uint32_t h[8];
  memcpy(h, c.h0, sizeof(h));
  const uint8_t* p = static_cast<const uint8_t*>(data);
  size_t left = n;
  while (left >= 64) {
    compress(h, p, c.k);
    p += 64;
    left -= 64;
  }
  // padding: 0x80, zeros to 56 mod 64, then the message length in bits (big-endian)
  uint8_t tail[128] = {};
  if (left) memcpy(tail, p, left);
  tail[left] = 0x80;
  const size_t len = left < 56 ? 64 : 128;
  const uint64_t bits = (uint64_t)n * 8;
  for (int i = 0; i < 8; ++i) tail[len - 1 - i] = (uint8_t)(bits >> (8 * i));
  compress(h, tail, c.k);
  if (len == 128) compress(h, tail + 64, c.k);
  for (int i = 0; i < 8; ++i) {
    out[4 * i] = (uint8_t)(h[i] >> 24);
    out[4 * i + 1] = (uint8_t)(h[i] >> 16);
    out[4 * i + 2] = (uint8_t)(h[i] >> 8);
    out[4 * i + 3] = (uint8_t)h[i];
  }
}

}  // namespace pa
