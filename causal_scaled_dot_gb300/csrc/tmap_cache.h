// tmap_cache.h -- a small least-recently-used cache of encoded TMA tensor maps.
//
// A tiled tensor map is a pure function of what the encoder is given: the base
// address, the element type, the extents, the strides and the box.  The key
// below holds every one of those inputs (strides follow from the extents for
// the contiguous views this library encodes) plus the device, so a hit always
// returns exactly the map a fresh encode would produce.  That makes the cache
// safe against reused addresses: a buffer that is freed and reallocated at the
// same address with the same geometry gets the same map, which is correct for
// it; any change of address, geometry or box is a different key.
//
// Not thread-safe by itself: the caller serialises lookup/insert (attn_api.cu
// holds a mutex around them).  Header-only and free of CUDA runtime calls, so
// host tests can compile it with a plain C++ compiler.
#pragma once

#include <cuda.h>

#include <cstdint>
#include <cstring>

namespace attn {

struct TmapKey {
    int device;
    const void* ptr;
    int elem_bytes;
    int D;
    int S;
    long long outer;
    int box_rows;

    bool operator==(const TmapKey& o) const {
        return device == o.device && ptr == o.ptr && elem_bytes == o.elem_bytes && D == o.D && S == o.S &&
               outer == o.outer && box_rows == o.box_rows;
    }
};

template <int N>
class TmapCache {
  public:
    // On a hit copies the cached map into *map and returns true.
    bool lookup(const TmapKey& key, CUtensorMap* map) {
        for (int i = 0; i < N; ++i) {
            if (used_[i] != 0 && keys_[i] == key) {
                std::memcpy(map, &maps_[i], sizeof(CUtensorMap));
                used_[i] = ++clock_;
                ++hits_;
                return true;
            }
        }
        ++misses_;
        return false;
    }
    // Stores a freshly encoded map, replacing the least recently used entry.
    void insert(const TmapKey& key, const CUtensorMap& map) {
        int victim = 0;
        for (int i = 0; i < N; ++i) {
            if (used_[i] == 0) {
                victim = i;
                break;
            }
            if (used_[i] < used_[victim]) victim = i;
        }
        keys_[victim] = key;
        std::memcpy(&maps_[victim], &map, sizeof(CUtensorMap));
        used_[victim] = ++clock_;
    }
    unsigned long long hits() const { return hits_; }
    unsigned long long misses() const { return misses_; }

  private:
    TmapKey keys_[N] = {};
    CUtensorMap maps_[N] = {};
    unsigned long long used_[N] = {};  // 0: empty slot; otherwise the last use's clock
    unsigned long long clock_ = 0;
    unsigned long long hits_ = 0, misses_ = 0;
};

}  // namespace attn
