// page_divisor.cpp -- the divisions the kernels take as a multiply-high and a
// shift, against the integer division:
//  * the paged cache's page index, floor(t / page_tokens) (with_page_divisor),
//    for every page size the library accepts up to 2^20 tokens (multiples of
//    128) and a set of large ones, at page boundaries and at random rows
//    below 2^31;
//  * the append kernels' group-index splits, floor(n / d) for 64-bit n
//    (make_fastdiv), for every d up to 4096, a set of large d, at multiples of
//    d, their neighbours and random n below 2^63.
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

static uint64_t next63() {
    const uint64_t hi = next31(), mid = next31(), lo = next31();
    return ((hi << 62) ^ (mid << 31) ^ lo) & 0x7FFFFFFFFFFFFFFFull;
}

static int check64(int32_t d, uint64_t n, long long* cases) {
    const tq::FastDiv f = tq::make_fastdiv(d);
    const uint64_t q =
        f.magic == 0 ? n : static_cast<uint64_t>((static_cast<unsigned __int128>(n) * f.magic) >> 64) >> f.shift;
    ++*cases;
    if (q != n / static_cast<uint64_t>(d)) {
        printf("d %d n %llu: %llu, want %llu\n", d, static_cast<unsigned long long>(n),
               static_cast<unsigned long long>(q), static_cast<unsigned long long>(n / static_cast<uint64_t>(d)));
        return 1;
    }
    return 0;
}

static int check_fastdiv(long long* cases) {
    const uint64_t top = 0x7FFFFFFFFFFFFFFFull;
    const int32_t big[] = {65535, 131072, 131071, 1000003, (1 << 30) + 1, 0x7FFFFFFF};
    for (int32_t d = 1; d <= 4096 + 6; ++d) {
        const int32_t dd = d <= 4096 ? d : big[d - 4097];
        const uint64_t last = top / static_cast<uint64_t>(dd) * static_cast<uint64_t>(dd);
        const uint64_t bounds[] = {0ull, static_cast<uint64_t>(dd), static_cast<uint64_t>(dd) * 1000003ull,
                                   last / 2 / static_cast<uint64_t>(dd) * static_cast<uint64_t>(dd), last};
        for (uint64_t b : bounds) {
            if (b > 0 && check64(dd, b - 1, cases)) return 1;
            if (check64(dd, b, cases)) return 1;
            if (b + dd - 1 <= top && check64(dd, b + dd - 1, cases)) return 1;
        }
        for (int i = 0; i < 200; ++i)
            if (check64(dd, next63(), cases) || check64(dd, next31(), cases)) return 1;
        if (check64(dd, top, cases)) return 1;
    }
    return 0;
}

int main() {
    long long cases = 0;
    if (check_fastdiv(&cases)) return 1;
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
