// A small cache of TMA descriptors for the grouped-GEMM launchers.  Encoding a
// CUtensorMap is host work on every call; a layer called again with the same
// buffers and shape (every decode step of a serving loop) reuses the encoded
// maps.  Keys are compared bytewise; the cache holds the last few entries.
#pragma once

#include <cuda.h>
#include <string.h>

#include <mutex>

namespace moe {

template <class Key, int NMaps, int Slots = 8>
class MapCache {
 public:
  // Copies the maps for `key` into `out` and returns true when cached.
  bool find(const Key& key, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < used_; ++i) {
      if (memcmp(&keys_[i], &key, sizeof(Key)) == 0) {
        memcpy(out, maps_[i], sizeof(CUtensorMap) * NMaps);
        return true;
      }
    }
    return false;
  }
  void put(const Key& key, const CUtensorMap* maps) {
    std::lock_guard<std::mutex> lock(mu_);
    const int i = used_ < Slots ? used_++ : next_;
    next_ = (i + 1) % Slots;
    memcpy(&keys_[i], &key, sizeof(Key));
    memcpy(maps_[i], maps, sizeof(CUtensorMap) * NMaps);
  }

 private:
  std::mutex mu_;
  Key keys_[Slots];
  CUtensorMap maps_[Slots][NMaps];
  int used_ = 0, next_ = 0;
};

}  // namespace moe
