"""Host-side checks of the library's own layout helpers (qmm_internal.cuh),
compiled as host code with nvcc and run on the CPU: the stream-K unit
partition and partial slots, the Q6_K lane geometry and code assembly, the
Q8_K planar permutation and the Q4_K header permutation. No GPU is used."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_quantized_matmul_q4_gb300", "csrc")

SRC = r'''
#include <cstdio>
#include <cstdlib>
#include <set>
#include "qmm_internal.cuh"
using namespace qmm;
#define CHECK(c) do { if (!(c)) { printf("FAIL %s line %d\n", #c, __LINE__); return 1; } } while (0)

int main() {
    // stream-K: unit u lies in the range of the CTA sk_cta_of names, for
    // unit counts above and below the grid (split K) alike
    const int64_t cases[][3] = {{344 * 16, 152, 16}, {128 * 32, 152, 32}, {32 * 16, 152, 16},
                                {4, 4, 2}, {256, 152, 256}, {7, 3, 7}, {1000 * 43, 152, 43}};
    for (auto &cs : cases) {
        const int64_t U = cs[0], G = cs[1], nsb = cs[2];
        for (int64_t u = 0; u < U; ++u) {
            const int64_t c = sk_cta_of(u, U, G);
            CHECK(c >= 0 && c < G && c * U / G <= u && u < (c + 1) * U / G);
        }
        // every CTA's pieces of its first and last tile get distinct slots
        std::set<int64_t> used;
        for (int64_t c = 0; c < G; ++c) {
            const int64_t u0 = c * U / G, u1 = (c + 1) * U / G;
            if (u1 <= u0) continue;
            const int64_t t0 = u0 / nsb, t1 = (u1 - 1) / nsb;
            const int64_t s0 = sk_slot(c, t0, U, G, nsb, 128), s1 = sk_slot(c, t1, U, G, nsb, 128);
            CHECK(s0 == c * 2 * 16384);
            CHECK(t0 == t1 || s1 == (c * 2 + 1) * 16384);
            CHECK(used.insert(s0).second);
            if (t1 != t0) CHECK(used.insert(s1).second);
        }
        // the fixup's shortcut: of a split tile's pieces only the first CTA's
        // can sit in slot 1 (the tile is that CTA's last), and only when the
        // CTA's range starts before the tile; every later CTA starts inside it
        for (int64_t t = 0; t < U / nsb; ++t) {
            const int64_t ca = sk_cta_of(t * nsb, U, G), cb = sk_cta_of(t * nsb + nsb - 1, U, G);
            for (int64_t c = ca; c <= cb && ca != cb; ++c)
                CHECK(sk_slot(c, t, U, G, nsb, 128) == (c * 2 + (c == ca && ca * U / G < t * nsb ? 1 : 0)) * 16384);
        }
    }
    // Q6_K lanes: (t, hi, i) covers the 256 elements once; the high-bit
    // positions of a lane word are 16 distinct bit pairs
    {
        std::set<int> e;
        for (int t = 0; t < 8; ++t)
            for (int hi = 0; hi < 2; ++hi)
                for (int i = 0; i < 16; ++i) CHECK(e.insert(q6k_elem(t, hi, i)).second);
        CHECK(e.size() == 256 && *e.begin() == 0 && *e.rbegin() == 255);
        std::set<int> b;
        for (int i = 0; i < 16; ++i) CHECK(b.insert(q6k_hbit_pos(i)).second && q6k_hbit_pos(i) % 2 == 0 &&
                                           q6k_hbit_pos(i) <= 30);
        // lane element i = 4w + k sits in byte k of ql word w: q6k_u puts its
        // high bits above its nibble
        srand(3);
        for (int trial = 0; trial < 200; ++trial) {
            int u[16];
            uint32_t hbits = 0, nib[4] = {0, 0, 0, 0};
            for (int i = 0; i < 16; ++i) {
                u[i] = rand() % 64;
                hbits |= (uint32_t)(u[i] >> 4) << q6k_hbit_pos(i);
                nib[i / 4] |= (uint32_t)((u[i] & 15) | ((rand() % 16) << 4)) << (8 * (i % 4));  // junk high nibble
            }
            for (int w = 0; w < 4; ++w) {
                const uint32_t got = q6k_u(nib[w], hbits, w);
                for (int k = 0; k < 4; ++k) CHECK((int)((got >> (8 * k)) & 255) == u[4 * w + k]);
            }
        }
    }
    // Q8_K planar order: the 32 lanes' 8-code groups fill the 256 bytes once,
    // and bsum word t holds the sums of the two groups lane slice t uses
    {
        std::set<int> off;
        for (int l = 0; l < 32; ++l)
            for (int k = 0; k < 8; ++k) CHECK(off.insert(q8K_code_offset(l) + k).second);
        CHECK(off.size() == 256 && *off.rbegin() == 255);
        std::set<int> bo;
        for (int b = 0; b < 16; ++b) CHECK(bo.insert(q8K_bsum_offset(b)).second && q8K_bsum_offset(b) < 32);
    }
    // Q4_K header: packed <-> canonical is a bijection on the 96 scale bits,
    // and field c carries (s_2c, m_2c, s_2c+1, m_2c+1)
    srand(5);
    for (int trial = 0; trial < 2000; ++trial) {
        uint4 h;
        h.x = (uint32_t)rand() ^ ((uint32_t)rand() << 16);
        h.y = (uint32_t)rand() ^ ((uint32_t)rand() << 16);
        h.z = (uint32_t)rand() ^ ((uint32_t)rand() << 16);
        h.w = (uint32_t)rand() ^ ((uint32_t)rand() << 16);
        const uint4 p = k4_header_to_packed(h);
        const uint4 back = k4_header_to_canonical(p);
        CHECK(back.x == h.x && back.y == h.y && back.z == h.z && back.w == h.w);
        int s[8], m[8];
        k4_scales_canonical(h, s, m);
        for (int c = 0; c < 4; ++c) {
            const uint32_t f = k4_field(p.y, p.z, p.w, c);
            CHECK((int)(f & 63) == s[2 * c] && (int)((f >> 6) & 63) == m[2 * c]);
            CHECK((int)((f >> 12) & 63) == s[2 * c + 1] && (int)((f >> 18) & 63) == m[2 * c + 1]);
        }
    }
    printf("OK\n");
    return 0;
}
'''


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not on PATH")
def test_host_layout_helpers(tmp_path):
    src = tmp_path / "geom.cu"
    src.write_text(SRC)
    exe = tmp_path / "geom"
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
           "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip().endswith("OK"), out.stdout[-2000:]
