/*
 * A plain C99 client of the W12 C ABI, host-side calls only (no GPU needed):
 * encode a small matrix with both window rules, validate, serialise, parse
 * the blob back, compare statistics, and check an unknown flag is refused.
 * Prints "ok" and exits 0 on success; any failure exits non-zero.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "w12.h"

#define CHECK(c)                                                          \
    do {                                                                  \
        if (!(c)) {                                                       \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
            return 1;                                                     \
        }                                                                 \
    } while (0)

int main(void)
{
    enum { N = 130, K = 300 };
    static uint16_t w[N * K];
    uint32_t s = 12345u;
    int i, mode;
    for (i = 0; i < N * K; i++) {
        s = s * 1664525u + 1013904223u;
        /* BF16 values around 2^-6 with a spread of exponents, a few zeros and one huge weight */
        w[i] = (uint16_t)(((s >> 31) << 15) | ((117u + ((s >> 8) % 9u)) << 7) | ((s >> 16) & 0x7Fu));
        if (i % 997 == 0)
            w[i] = 0;
    }
    w[7] = 0x7F00;
    for (mode = 0; mode < 2; mode++) {
        w12_host *h = NULL, *h2 = NULL;
        w12_stats st, st2;
        size_t len = 0, len2 = 0;
        uint8_t *blob;
        CHECK(w12_encode_ex(w, N, K, 2, mode ? W12_ENCODE_COUNT_MAX : 0u, &h) == W12_OK);
        CHECK(w12_validate(h) == W12_OK);
        CHECK(w12_serialize(h, NULL, 0, &len) == W12_OK && len > 0);
        blob = (uint8_t *)malloc(len);
        CHECK(blob != NULL);
        CHECK(w12_serialize(h, blob, len, &len2) == W12_OK && len2 == len);
        CHECK(memcmp(blob, "W12", 4) == 0);
        CHECK(w12_deserialize(blob, len, &h2) == W12_OK);
        CHECK(w12_host_stats(h, &st) == W12_OK && w12_host_stats(h2, &st2) == W12_OK);
        CHECK(st.N == N && st.K == K && st2.n_escapes == st.n_escapes && st.n_escapes > 0);
        printf("window rule %d: %lld escapes, %zu bytes\n", mode, (long long)st.n_escapes, len);
        free(blob);
        w12_host_free(h);
        w12_host_free(h2);
    }
    {
        w12_host *h = NULL;
        CHECK(w12_encode_ex(w, N, K, 0, 0x80u, &h) == W12_ERR_INVALID_ARG && h == NULL);
        CHECK(strlen(w12_status_string(W12_ERR_CORRUPT)) > 0);
    }
    printf("ok\n");
    return 0;
}
