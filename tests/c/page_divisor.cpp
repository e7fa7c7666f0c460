// page_divisor.cpp -- the paged cache's page index, floor(t / page_tokens),
// computed as the kernels do (multiply-high by the reciprocal that
// with_page_divisor derives, then a shift), against the integer division for
// every page size the library accepts up to 2^20 tokens (multiples of 128) and
// a set of large ones, at every page boundary and at random rows below 2^31.
// Prints "OK <cases>" and exits 0, or the first mismatch and exits 1.
#include <stdint.h>
#include <stdio.h>

#include "tq_internal.h"

static uint64_t rng = 0x2545F4914F6CDD1Dull;
static uint32_t next31() {
    rng ^= rng << 13;
    rng ^= rng >> 7;
    rng ^= rng << 17;
    return static_cast<uint32_t>(rng >> 33);  // 31 bits
}

static int check(int32_t d, uint32_t t, long long* cases) {
    tq::RowMap m{nullptr, d, 1, 1, 0, 0};
    m = tq::with_page_divisor(m);
    const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(t) * m.page_magic) >> 32);
    const uint32_t q = hi >> m.page_shift;
    ++*cases;
    if (q != t / static_cast<uint32_t>(d)) {
        printf("page_tokens %d row %u: %u, want %u\n", d, t, q, t / static_cast<uint32_t>(d));
        return 1;
    }
    return 0;
}

int main() {
    long long cases = 0;
    const uint32_t top = 0x7FFFFFFFu;
    for (int32_t d = 128; d <= (1 << 20); d += 128) {
        // both sides of the first, a middle and the last page boundaries
        const uint32_t last = top / d * d;
        const uint32_t bounds[] = {0u, static_cast<uint32_t>(d), static_cast<uint32_t>(d) * 7u, last / 2 / d * d, last};
        for (uint32_t b : bounds) {
            if (b > 0 && check(d, b - 1, &cases)) return 1;
            if (check(d, b, &cases)) return 1;
            if (b + d - 1 <= top && check(d, b + d - 1, &cases)) return 1;
        }
        for (int i = 0; i < 64; ++i)
            if (check(d, next31(), &cases)) return 1;
        if (check(d, top, &cases)) return 1;
    }
    const int32_t big[] = {(1 << 20) + 128, 3 << 20, 1000000 * 128, 0x7FFFFF80};
    for (int32_t d : big) {
        for (uint32_t k = 0; k <= top / d; ++k) {
            const uint32_t b = k * static_cast<uint32_t>(d);
            if (b > 0 && check(d, b - 1, &cases)) return 1;
            if (check(d, b, &cases)) return 1;
        }
        for (int i = 0; i < 100000; ++i)
            if (check(d, next31(), &cases)) return 1;
        if (check(d, top, &cases)) return 1;
    }
    printf("OK %lld\n", cases);
    return 0;
}
