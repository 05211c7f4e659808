// CPU check of the per-stream workspace arenas (paged_kv_decode_19_gb300/csrc/arena.h)
// with fake stream-ordered operations that log every call: streams get separate
// buffers; growth allocates the new buffer before it releases the old one, releases it
// on the same stream, and zero-fills new counters; a failed allocation leaves the arena
// as it was; release frees both buffers once; during stream capture the arena is found
// by the stream handle that last used it, handed out without any call, and a handle that
// came back with a new stream finds the new stream's arena.
#include <stdio.h>
#include <stdlib.h>

#include <string>
#include <vector>

#include "arena.h"

struct Call {
  std::string op;
  size_t id;       // buffer id (1-based allocation index)
  size_t bytes;
  void* stream;
};
struct Fake {
  std::vector<Call> log;
  std::vector<char*> bufs;
  std::vector<bool> live;
  int fail_next_alloc = 0;
};

static size_t id_of(Fake* f, void* p) {
  for (size_t i = 0; i < f->bufs.size(); ++i)
    if (f->bufs[i] == p) return i + 1;
  return 0;
}
static int f_alloc(void* ctx, void** p, size_t bytes, void* st) {
  Fake* f = (Fake*)ctx;
  if (f->fail_next_alloc) {
    f->fail_next_alloc = 0;
    return 2;
  }
  char* b = (char*)malloc(bytes);
  f->bufs.push_back(b);
  f->live.push_back(true);
  *p = b;
  f->log.push_back({"alloc", f->bufs.size(), bytes, st});
  return 0;
}
static int f_release(void* ctx, void* p, void* st) {
  Fake* f = (Fake*)ctx;
  const size_t id = id_of(f, p);
  if (!id || !f->live[id - 1]) return 1;  // unknown or double free
  f->live[id - 1] = false;
  f->log.push_back({"release", id, 0, st});
  return 0;
}
static int f_zero(void* ctx, void* p, size_t bytes, void* st) {
  Fake* f = (Fake*)ctx;
  f->log.push_back({"zero", id_of(f, p), bytes, st});
  return 0;
}

static int failures = 0;
#define CHECK(c)                                             \
  do {                                                       \
    if (!(c)) {                                              \
      fprintf(stderr, "FAILED line %d: %s\n", __LINE__, #c); \
      ++failures;                                            \
    }                                                        \
  } while (0)

int main() {
  Fake f;
  pd::ArenaOps ops = {&f, f_alloc, f_release, f_zero};
  pd::ArenaTable t;
  void* sA = (void*)0x10;
  void* sB = (void*)0x20;
  void *cA, *pA, *cB, *pB;
  // first use of stream A: counters allocated and zeroed on A, partials allocated on A
  CHECK(t.acquire(7, sA, 1000, 5000, ops, &cA, &pA) == 0);
  CHECK(f.log.size() == 3 && f.log[0].op == "alloc" && f.log[1].op == "zero" &&
        f.log[1].id == f.log[0].id && f.log[2].op == "alloc");
  for (const Call& c : f.log) CHECK(c.stream == sA);
  CHECK(f.log[0].bytes >= 1000 && f.log[1].bytes == f.log[0].bytes && f.log[2].bytes >= 5000);
  // same size again: no new calls, same buffers
  void *c2, *p2;
  CHECK(t.acquire(7, sA, 1000, 5000, ops, &c2, &p2) == 0);
  CHECK(f.log.size() == 3 && c2 == cA && p2 == pA);
  // stream B: its own buffers, nothing of A's touched
  CHECK(t.acquire(9, sB, 1000, 5000, ops, &cB, &pB) == 0);
  CHECK(cB != cA && pB != pA && t.size() == 2 && f.log.size() == 6);
  for (size_t i = 3; i < 6; ++i) CHECK(f.log[i].stream == sB);
  // growth of A's partials: the new buffer first, then the old one released on A
  const size_t n0 = f.log.size();
  void *c3, *p3;
  CHECK(t.acquire(7, sA, 1000, 1 << 22, ops, &c3, &p3) == 0);
  CHECK(c3 == cA && p3 != pA);
  CHECK(f.log.size() == n0 + 2 && f.log[n0].op == "alloc" && f.log[n0 + 1].op == "release" &&
        f.log[n0 + 1].id == id_of(&f, pA) && f.log[n0 + 1].stream == sA);
  // growth of A's counters: new buffer allocated, zeroed, then the old one released
  const size_t n1 = f.log.size();
  void *c4, *p4;
  CHECK(t.acquire(7, sA, 1 << 16, 1 << 22, ops, &c4, &p4) == 0);
  CHECK(c4 != cA && p4 == p3);
  CHECK(f.log.size() == n1 + 3 && f.log[n1].op == "alloc" && f.log[n1 + 1].op == "zero" &&
        f.log[n1 + 1].id == f.log[n1].id && f.log[n1 + 2].op == "release" &&
        f.log[n1 + 2].id == id_of(&f, cA));
  // stream capture: the arena last used by the handle, handed out as it is (no calls);
  // a need beyond its size, or a handle never seen, gives kNoRoom
  {
    const size_t nc = f.log.size();
    void *cc = nullptr, *pc = nullptr;
    CHECK(t.acquire_captured(sA, 1 << 16, 1 << 22, &cc, &pc) == 0 && cc == c4 && pc == p3);
    CHECK(t.acquire_captured(sA, 1 << 16, 1 << 27, &cc, &pc) == pd::ArenaTable::kNoRoom);
    CHECK(t.acquire_captured((void*)0x99, 16, 16, &cc, &pc) == pd::ArenaTable::kNoRoom);
    CHECK(t.acquire_captured(nullptr, 16, 16, &cc, &pc) == pd::ArenaTable::kNoRoom);
    CHECK(f.log.size() == nc);
    // a new stream (id 11) that got stream B's handle back: the handle now finds its arena
    void *c11, *p11;
    CHECK(t.acquire(11, sB, 1000, 5000, ops, &c11, &p11) == 0 && c11 != cB);
    CHECK(t.acquire_captured(sB, 16, 16, &cc, &pc) == 0 && cc == c11 && pc == p11);
    CHECK(t.release(11, sB, ops) == 0);
    CHECK(t.acquire_captured(sB, 16, 16, &cc, &pc) == pd::ArenaTable::kNoRoom);
  }
  // a failed allocation while growing: error returned, the arena keeps its buffers
  f.fail_next_alloc = 1;
  void *c5 = nullptr, *p5 = nullptr;
  CHECK(t.acquire(7, sA, 1 << 16, 1 << 26, ops, &c5, &p5) == 2);
  const pd::Arena* a = t.find_const(7);
  CHECK(a && a->cnt == c4 && a->part == p3 && f.live[id_of(&f, p3) - 1]);
  // release: both buffers of A freed once on A; B untouched; unknown key is a no-op
  CHECK(t.release(7, sA, ops) == 0);
  CHECK(t.size() == 1 && !f.live[id_of(&f, c4) - 1] && !f.live[id_of(&f, p3) - 1]);
  CHECK(f.live[id_of(&f, cB) - 1] && f.live[id_of(&f, pB) - 1]);
  CHECK(t.release(7, sA, ops) == 0 && t.release(12345, sA, ops) == 0);
  // every buffer ever handed out to A is released exactly once, none of B's
  size_t live = 0;
  for (bool l : f.live) live += l ? 1 : 0;
  CHECK(live == 2);
  if (failures) return 1;
  printf("arena bookkeeping ok\n");
  return 0;
}
