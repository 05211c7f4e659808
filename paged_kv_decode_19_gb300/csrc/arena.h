// Per-stream arenas of the library-managed decode workspace (host code only, no CUDA
// headers: the allocator calls come in through ArenaOps, so the bookkeeping is tested
// on the CPU with fake operations).
//
// Why per stream: a split decode uses its workspace's arrival counters and partial
// (out, lse) slots from the launch until the kernel ends.  Two decodes in flight on
// different streams must therefore never share one workspace.  Each stream (keyed by
// its process-unique CUDA stream id) gets its own arena, used only by work enqueued on
// that stream, so calls on one stream are ordered by the stream itself.
//
// Why stream-ordered growth: a buffer that is too small is never freed at once (a
// kernel enqueued earlier on the stream may still read it).  The larger buffer is
// allocated first, then the old one is released with a stream-ordered free, which runs
// only after all work enqueued before it on that stream.  A new counter buffer is
// zero-filled on the stream before first use; every completed decode leaves its
// counters at zero again.
//
// The caller serialises acquire/release and the enqueue of the kernel that uses the
// returned buffers (one mutex per device), so no other host thread can retire a
// buffer between its hand-out and the launch that uses it.
//
// Stream capture (CUDA graphs): a capturing stream's id cannot be queried, and memory
// must not be allocated or freed behind the graph's back, so acquire_captured finds the
// arena by the stream handle that last used it outside capture and hands out its
// buffers as they are; it never allocates.  The graph then owns references to those
// buffers: they stay valid until the stream's arena is released or grows.
#pragma once

#include <stddef.h>

#include <vector>

namespace pd {

// Stream-ordered device memory operations (0 = success, anything else = an error code
// returned unchanged to the caller).
struct ArenaOps {
  void* ctx;
  int (*alloc)(void* ctx, void** ptr, size_t bytes, void* stream);
  int (*release)(void* ctx, void* ptr, void* stream);
  int (*zero)(void* ctx, void* ptr, size_t bytes, void* stream);
};

struct Arena {
  unsigned long long key;  // stream id
  void* handle = nullptr;  // the stream handle of its last acquire (null: superseded)
  void* cnt = nullptr;     // arrival counters (zero between calls)
  size_t cnt_bytes = 0;
  void* part = nullptr;    // partial (lse, out) slots
  size_t part_bytes = 0;
};

class ArenaTable {
 public:
  static constexpr size_t kCntGrain = 4096;
  static constexpr size_t kPartGrain = size_t(1) << 20;

  // Buffers of at least cnt_need / part_need bytes for work on `stream` (key = its
  // id): the arena's current ones, or larger ones allocated now (the old ones released
  // stream-ordered).  On an error nothing of the arena changes except what was
  // already swapped in.
  int acquire(unsigned long long key, void* stream, size_t cnt_need, size_t part_need,
              const ArenaOps& ops, void** cnt, void** part) {
    Arena* a = find(key);
    if (!a) {
      arenas_.push_back(Arena{});
      a = &arenas_.back();
      a->key = key;
    }
    // a handle names one live stream at a time: an older arena that saw it (a destroyed
    // stream whose handle came back) is no longer found by it
    for (Arena& o : arenas_)
      if (&o != a && o.handle == stream) o.handle = nullptr;
    a->handle = stream;
    if (a->cnt_bytes < cnt_need) {
      const size_t bytes = round_up(cnt_need * 2, kCntGrain);
      void* p = nullptr;
      int e = ops.alloc(ops.ctx, &p, bytes, stream);
      if (e) return e;
      e = ops.zero(ops.ctx, p, bytes, stream);
      if (e) {
        ops.release(ops.ctx, p, stream);
        return e;
      }
      if (a->cnt) {
        e = ops.release(ops.ctx, a->cnt, stream);
        if (e) {
          ops.release(ops.ctx, p, stream);
          return e;
        }
      }
      a->cnt = p;
      a->cnt_bytes = bytes;
    }
    if (a->part_bytes < part_need) {
      const size_t bytes = round_up(part_need + part_need / 4, kPartGrain);
      void* p = nullptr;
      int e = ops.alloc(ops.ctx, &p, bytes, stream);
      if (e) return e;
      if (a->part) {
        e = ops.release(ops.ctx, a->part, stream);
        if (e) {
          ops.release(ops.ctx, p, stream);
          return e;
        }
      }
      a->part = p;
      a->part_bytes = bytes;
    }
    *cnt = a->cnt;
    *part = a->part;
    return 0;
  }

  // During stream capture: the buffers of the arena last acquired with `stream`, if it
  // holds cnt_need / part_need bytes; else kNoRoom (nothing is allocated).
  static constexpr int kNoRoom = -1;
  int acquire_captured(void* stream, size_t cnt_need, size_t part_need, void** cnt,
                       void** part) const {
    for (const Arena& a : arenas_) {
      if (a.handle != stream || !stream) continue;
      if (a.cnt_bytes < cnt_need || a.part_bytes < part_need) return kNoRoom;
      *cnt = a.cnt;
      *part = a.part;
      return 0;
    }
    return kNoRoom;
  }
  // Releases the arena of stream `key` (stream-ordered) and forgets it; no arena: 0.
  int release(unsigned long long key, void* stream, const ArenaOps& ops) {
    for (size_t i = 0; i < arenas_.size(); ++i) {
      if (arenas_[i].key != key) continue;
      int e = 0;
      if (arenas_[i].cnt) e = ops.release(ops.ctx, arenas_[i].cnt, stream);
      if (arenas_[i].part) {
        const int e2 = ops.release(ops.ctx, arenas_[i].part, stream);
        if (!e) e = e2;
      }
      arenas_.erase(arenas_.begin() + (long)i);
      return e;
    }
    return 0;
  }

  size_t size() const { return arenas_.size(); }
  const Arena* find_const(unsigned long long key) const {
    for (const Arena& a : arenas_)
      if (a.key == key) return &a;
    return nullptr;
  }

 private:
  static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
  Arena* find(unsigned long long key) {
    for (Arena& a : arenas_)
      if (a.key == key) return &a;
    return nullptr;
  }
  std::vector<Arena> arenas_;
};

}  // namespace pd
