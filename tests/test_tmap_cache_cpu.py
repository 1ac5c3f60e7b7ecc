"""The host-side cache of encoded TMA tensor maps (csrc/tmap_cache.h), compiled
on its own with g++ and driven by a small C++ program: hits return exactly
what was stored, every change of address or geometry misses, a reused address
with the same geometry maps to the same (correct) tensor map, and the least
recently used entry is the one replaced.  No GPU and no CUDA runtime call."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "causal_scaled_dot_gb300", "csrc")

PROGRAM = r"""
#include "tmap_cache.h"
#include <cstdio>
#include <cstring>

using attn::TmapCache;
using attn::TmapKey;

// Stand-in for the driver's encoder: a deterministic function of the key, so
// that a cached map can be compared with what a fresh encode would give.
static CUtensorMap fake_encode(const TmapKey& k) {
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    unsigned long long w[6] = {(unsigned long long)(size_t)k.ptr, (unsigned long long)k.device,
                               (unsigned long long)k.elem_bytes, (unsigned long long)k.D,
                               (unsigned long long)k.S * 1000003ull + (unsigned long long)k.outer,
                               (unsigned long long)k.box_rows};
    std::memcpy(&m, w, sizeof w);
    return m;
}
static bool same(const CUtensorMap& a, const CUtensorMap& b) { return std::memcmp(&a, &b, sizeof a) == 0; }

#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

int main() {
    TmapCache<4> c;
    const void* p = reinterpret_cast<const void*>(0x7f0000001000ull);
    TmapKey k{0, p, 2, 128, 4096, 64, 128};
    CUtensorMap got;
    CHECK(!c.lookup(k, &got));                       // empty: miss
    c.insert(k, fake_encode(k));
    CHECK(c.lookup(k, &got) && same(got, fake_encode(k)));

    // every input of the encode is part of the key
    TmapKey v[7] = {k, k, k, k, k, k, k};
    v[0].device = 1; v[1].ptr = reinterpret_cast<const void*>(0x7f0000002000ull); v[2].elem_bytes = 1;
    v[3].D = 64; v[4].S = 4095; v[5].outer = 65; v[6].box_rows = 32;
    for (int i = 0; i < 7; ++i) CHECK(!c.lookup(v[i], &got));

    // a buffer freed and reallocated at the same address with the same
    // geometry has the same key: the hit is the map a fresh encode gives
    TmapKey reused = k;
    CHECK(c.lookup(reused, &got) && same(got, fake_encode(reused)));

    // a changed shape at the same address misses, and once inserted both live
    TmapKey reshaped = k; reshaped.S = 2048; reshaped.outer = 128;
    CHECK(!c.lookup(reshaped, &got));
    c.insert(reshaped, fake_encode(reshaped));
    CHECK(c.lookup(reshaped, &got) && same(got, fake_encode(reshaped)));
    CHECK(c.lookup(k, &got) && same(got, fake_encode(k)));

    // least recently used replacement: fill to capacity, touch k, add one more
    TmapKey a = k; a.ptr = reinterpret_cast<const void*>(0x1000ull);
    TmapKey b = k; b.ptr = reinterpret_cast<const void*>(0x2000ull);
    c.insert(a, fake_encode(a));
    c.insert(b, fake_encode(b));                    // holds k, reshaped, a, b
    CHECK(c.lookup(reshaped, &got));
    CHECK(c.lookup(k, &got));                        // a is now the oldest
    TmapKey d = k; d.ptr = reinterpret_cast<const void*>(0x3000ull);
    c.insert(d, fake_encode(d));
    CHECK(!c.lookup(a, &got));
    CHECK(c.lookup(b, &got) && same(got, fake_encode(b)));
    CHECK(c.lookup(d, &got) && same(got, fake_encode(d)));
    CHECK(c.lookup(k, &got) && same(got, fake_encode(k)));
    std::printf("OK hits=%llu misses=%llu\n", c.hits(), c.misses());
    return 0;
}
"""


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        inc = os.path.join(cand, "include") if cand else ""
        if inc and os.path.exists(os.path.join(inc, "cuda.h")):
            return inc
    nvcc = shutil.which("nvcc")
    if nvcc:
        inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
        if os.path.exists(os.path.join(inc, "cuda.h")):
            return inc
    return None


def test_tensor_map_cache_hits_misses_and_replacement(tmp_path):
    inc = _cuda_include()
    if inc is None or shutil.which("g++") is None:
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "cache_test.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "cache_test"
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", "-I", CSRC, "-I", inc, "-o", str(exe), str(src)],
                   check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.startswith("OK")
