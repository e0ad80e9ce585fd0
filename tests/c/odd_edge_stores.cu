// Host check of the odd-start kernel's edge store sequences: for every
// element range [lo, hi) an edge lane can store (lo = 0 or 1, hi odd or the
// whole vector) and every vector width, the sequence writes exactly the
// range's bytes, each from the right word.  Prints "ok <cases>" or the
// first failure.
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "rope_kernels.cuh"

template <int E, int V>
static int check_width() {
    constexpr int W = V / 4, VE = V / E;
    int cases = 0;
    alignas(16) unsigned char buf[64];
    uint32_t sw[W];
    for (int k = 0; k < W; ++k) sw[k] = 0x11111111u * uint32_t(k + 1) + 0x01020304u;
    const unsigned char* src = reinterpret_cast<const unsigned char*>(sw);
    for (int lo = 0; lo <= 1; ++lo) {
        for (int hi = 1; hi <= VE; ++hi) {
            // hi is odd and leaves at least one pair, or the vector's end
            if (!((hi & 1) ? hi >= 3 : hi == VE)) continue;
            memset(buf, 0xEE, sizeof(buf));
            char* p = reinterpret_cast<char*>(buf + 16);
            if (E == 2)
                rope::store_span_lo<uint16_t, VE>(p, sw, lo, hi);
            else
                rope::store_span_lo<float, VE>(p, sw, lo, hi);
            for (int byte = 0; byte < (int)sizeof(buf); ++byte) {
                const int off = byte - 16;
                const bool in = off >= lo * E && off < hi * E;
                const unsigned char want = in ? src[off] : 0xEE;
                if (buf[byte] != want) {
                    printf("FAIL e=%d V=%d lo=%d hi=%d byte %d: got %02x want %02x\n", E, V, lo, hi,
                           off, buf[byte], want);
                    return -1;
                }
            }
            ++cases;
        }
    }
    return cases;
}

int main() {
    const int r[] = {check_width<2, 16>(), check_width<2, 8>(), check_width<4, 16>(),
                     check_width<4, 8>()};
    int total = 0;
    for (int c : r) {
        if (c < 0) return 1;
        total += c;
    }
    printf("ok %d\n", total);
    return 0;
}
