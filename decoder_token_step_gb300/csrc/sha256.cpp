// sha256.cpp -- SHA-256 of a definition text (host). "Local inference and architectures", section
// "What is in effect right now": every definition is identified by the sha256 of its text, so two
// runs with the same sha ran the same architecture.
//
// Written from the Secure Hash Standard (FIPS 180-4, section 6.2). The round constants and the
// initial hash value are derived here exactly as the standard defines them -- the first 32 bits of
// the fractional parts of the cube roots of the first 64 primes, and of the square roots of the
// first 8 primes -- by integer root refinement, rather than copied as a table.
#include <cstdint>
#include <cstring>
#include <string>

#include "syn_internal.h"

namespace syn {

namespace {

using u128 = unsigned __int128;

// first 32 fractional bits of the k-th root (k = 2 or 3) of p: the largest a with a^k <= p * 2^(32k),
// reduced modulo 2^32 (drops the integer part)
uint32_t frac_root_bits(uint32_t p, int k) {
    const u128 target = (u128)p << (32 * k);
    uint64_t lo = 0, hi = (uint64_t)1 << 40;   // roots of primes < 400 are below 2^9 * 2^32
    while (hi - lo > 1) {
        const uint64_t mid = lo + (hi - lo) / 2;
        u128 v = mid;
        for (int i = 1; i < k; ++i) v *= mid;
        if (v <= target) lo = mid;
        else hi = mid;
    }
    return (uint32_t)lo;
}

struct Tables {
    uint32_t k[64], h0[8];
    Tables() {
        int n = 0;
        for (uint32_t c = 2; n < 64; ++c) {
            bool prime = true;
            for (uint32_t d = 2; d * d <= c; ++d)
                if (c % d == 0) { prime = false; break; }
            if (!prime) continue;
            k[n] = frac_root_bits(c, 3);
            if (n < 8) h0[n] = frac_root_bits(c, 2);
            ++n;
        }
    }
};

const Tables &tables() {
    static const Tables t;
    return t;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void compress(uint32_t (&h)[8], const uint8_t *block, const uint32_t (&k)[64]) {
    uint32_t w[64];
    for (int t = 0; t < 16; ++t)
        w[t] = (uint32_t)block[4 * t] << 24 | (uint32_t)block[4 * t + 1] << 16 | (uint32_t)block[4 * t + 2] << 8 | block[4 * t + 3];
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
        hh = g; g = f; f = e; e = d + t1; d = c; c = b; b = a; a = t1 + t2;
    }
    h[0] += a; h[1] += b; h[2] += c; h[3] += d; h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
}

}  // namespace

std::string sha256_hex(const void *data, size_t len) {
    const Tables &T = tables();
    uint32_t h[8];
    std::memcpy(h, T.h0, sizeof h);
    const uint8_t *p = static_cast<const uint8_t *>(data);
    size_t off = 0;
    for (; off + 64 <= len; off += 64) compress(h, p + off, T.k);
    // padding: a 1 bit, zeros, then the message length in bits as a 64-bit big-endian integer
    uint8_t tail[128] = {};
    const size_t rem = len - off;
    if (rem) std::memcpy(tail, p + off, rem);
    tail[rem] = 0x80;
    const size_t tail_len = rem + 9 <= 64 ? 64 : 128;
    const uint64_t bits = (uint64_t)len * 8;
    for (int i = 0; i < 8; ++i) tail[tail_len - 1 - i] = (uint8_t)(bits >> (8 * i));
    compress(h, tail, T.k);
    if (tail_len == 128) compress(h, tail + 64, T.k);
    static const char *hexd = "0123456789abcdef";
    std::string out(64, '0');
    for (int i = 0; i < 8; ++i)
        for (int j = 0; j < 8; ++j) out[8 * i + j] = hexd[(h[i] >> (28 - 4 * j)) & 15];
    return out;
}

}  // namespace syn
