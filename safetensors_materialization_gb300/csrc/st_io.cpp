// st_io.cpp -- range reads of safetensors shard files into host memory.
//
// "Disk tier safetensors streaming design audit (ComfyUI)", "Range reads and
// tiering": a tensor's bytes are read from disk into (optionally pinned) host
// memory and copied to the GPU, without reading the rest of the file.  Here a
// set of shard files is addressed as one arena (the layout st_index_concat
// gives): arena byte x of part k lives at file offset offset_k + (x - base_k).
// Reads use pread on host threads; the disk -> pinned -> device -> materialize
// pipeline built on them is st_load_files (st_plan.cpp).  Each file is also
// mapped read-only, so that on hosts whose GPU reads pageable memory through
// the host's page tables a chunk can be copied to the device straight from
// the page cache, with no CPU copy (st_load_files without a ring).
#include <cuda_runtime_api.h>
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <cerrno>
#include <condition_variable>
#include <deque>
#include <functional>
#include <mutex>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "st_internal.h"

// Reader threads kept for the lifetime of a files object (started on first
// use, at most kMaxReaders): a range read hands each thread one span and
// waits for all of them.  Starting threads for every read cost a third of
// the page-cache read rate.
struct ReaderPool {
  static constexpr uint32_t kMaxReaders = 32;
  std::mutex m;
  std::condition_variable cv;
  std::deque<std::function<void()>> jobs;
  std::vector<std::thread> threads;
  bool stop = false;
  // Grows to n threads (fewer if threads cannot be started).
  void ensure(uint32_t n) {
    std::lock_guard<std::mutex> g(m);
    n = std::min(n, kMaxReaders);
    try {
      while (threads.size() < n)
        threads.emplace_back([this] {
          for (;;) {
            std::function<void()> job;
            {
              std::unique_lock<std::mutex> lk(m);
              cv.wait(lk, [this] { return stop || !jobs.empty(); });
              if (jobs.empty()) return;  // stop, nothing left
              job = std::move(jobs.front());
              jobs.pop_front();
            }
            job();
          }
        });
    } catch (const std::exception &) {
    }
  }
  // Runs every job of the batch (on the pool, or here when it has no
  // threads) and returns when all are done.
  void run(std::vector<std::function<void()>> &batch) {
    bool pooled;
    {
      std::lock_guard<std::mutex> g(m);
      pooled = !threads.empty();
    }
    if (!pooled) {
      for (auto &job : batch) job();
      return;
    }
    std::mutex dm;
    std::condition_variable dcv;
    size_t left = batch.size(), queued = 0;
    {
      std::lock_guard<std::mutex> g(m);
      try {
        for (auto &job : batch) {
          jobs.emplace_back([&dm, &dcv, &left, job] {
            job();
            std::lock_guard<std::mutex> dg(dm);  // notify under the lock: the waiter
            if (--left == 0) dcv.notify_all();   // cannot return (and drop dm/dcv) before
          });
          ++queued;
        }
      } catch (const std::bad_alloc &) {
        // the jobs not queued run here, below
      }
    }
    cv.notify_all();
    for (size_t i = queued; i < batch.size(); ++i) batch[i]();
    std::unique_lock<std::mutex> lk(dm);
    left -= batch.size() - queued;
    dcv.wait(lk, [&] { return left == 0; });
  }
  ~ReaderPool() {
    {
      std::lock_guard<std::mutex> g(m);
      stop = true;
    }
    cv.notify_all();
    for (auto &t : threads) t.join();
  }
};

struct st_files_s {
  struct Part {
    std::string path;
    int fd = -1;
    uint64_t offset = 0, bytes = 0, base = 0;
    const uint8_t *map = nullptr;  // the whole file, PROT_READ / MAP_SHARED; NULL if mapping failed
    uint64_t map_bytes = 0;
  };
  std::vector<Part> parts;  // sorted by base, non-overlapping
  uint64_t arena_bytes = 0;
  uint64_t uid = 0;  // unique in the process: RAM-tier entries are keyed by it, not by the address
  mutable ReaderPool readers;
  ~st_files_s() {
    for (Part &p : parts) {
      if (p.map) munmap(const_cast<uint8_t *>(p.map), p.map_bytes);
      if (p.fd >= 0) close(p.fd);
    }
  }
};

namespace stmat {

namespace {

// pread until `n` bytes arrived; false on an error or end of file.
bool pread_all(int fd, uint8_t *dst, uint64_t n, uint64_t off, int *err) {
  while (n) {
    const size_t want = static_cast<size_t>(std::min<uint64_t>(n, 1ull << 30));
    const ssize_t got = pread(fd, dst, want, static_cast<off_t>(off));
    if (got < 0) {
      if (errno == EINTR) continue;
      *err = errno;
      return false;
    }
    if (got == 0) {
      *err = 0;  // the file ended early
      return false;
    }
    dst += got;
    off += static_cast<uint64_t>(got);
    n -= static_cast<uint64_t>(got);
  }
  return true;
}

// Arena bytes [lo, hi) into host + (lo - begin), one thread's share.
bool read_span(const st_files_s &f, uint64_t begin, uint64_t lo, uint64_t hi, uint8_t *host, std::string *msg) {
  for (const auto &p : f.parts) {
    const uint64_t a = std::max(lo, p.base), b = std::min(hi, p.base + p.bytes);
    if (a >= b) continue;
    int err = 0;
    if (!pread_all(p.fd, host + (a - begin), b - a, p.offset + (a - p.base), &err)) {
      *msg = "reading " + std::to_string(b - a) + " bytes at " + std::to_string(p.offset + (a - p.base)) + " of " +
             p.path + ": " + (err ? std::strerror(err) : "the file ended early");
      return false;
    }
  }
  return true;
}

}  // namespace

st_status read_arena(const st_files_s *f, uint64_t begin, uint64_t bytes, void *host, uint32_t threads) {
  if (!f || (bytes && !host)) return set_error(ST_E_INVAL, "NULL argument");
  if (begin > f->arena_bytes || bytes > f->arena_bytes - begin)
    return set_error(ST_E_INVAL, "range %llu + %llu is beyond the %llu-byte arena", (unsigned long long)begin,
                     (unsigned long long)bytes, (unsigned long long)f->arena_bytes);
  if (!bytes) return ST_OK;
  uint8_t *dst = static_cast<uint8_t *>(host);
  // Split in up to `threads` spans of whole 1 MiB blocks.
  constexpr uint64_t kBlock = 1ull << 20;
  const uint64_t blocks = (bytes + kBlock - 1) / kBlock;
  const uint32_t t = static_cast<uint32_t>(std::max<uint64_t>(1, std::min<uint64_t>(threads ? threads : 1, blocks)));
  if (t == 1) {
    std::string msg;
    if (!read_span(*f, begin, begin, begin + bytes, dst, &msg)) return set_error(ST_E_IO, "%s", msg.c_str());
    return ST_OK;
  }
  std::vector<std::string> msgs(t);
  std::atomic<bool> ok{true};
  try {
    std::vector<std::function<void()>> batch;
    for (uint32_t i = 0; i < t; ++i) {
      const uint64_t lo = begin + std::min(bytes, blocks * i / t * kBlock);
      const uint64_t hi = begin + std::min(bytes, blocks * (i + 1) / t * kBlock);
      batch.emplace_back([&, i, lo, hi] {
        if (!read_span(*f, begin, lo, hi, dst, &msgs[i])) ok = false;
      });
    }
    f->readers.ensure(t);
    f->readers.run(batch);
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "queueing %u reads", t);
  }
  if (!ok) {
    for (const auto &m : msgs)
      if (!m.empty()) return set_error(ST_E_IO, "%s", m.c_str());
  }
  return ST_OK;
}

uint64_t files_arena_bytes(const st_files_s *f) { return f->arena_bytes; }

bool files_mapped(const st_files_s *f) {
  for (const auto &p : f->parts)
    if (!p.map && p.bytes) return false;
  return true;
}

namespace {

#ifndef MADV_POPULATE_READ
#define MADV_POPULATE_READ 22  // Linux 5.14
#endif

// Faults arena bytes [begin, end) of the files' mappings into the process's
// page tables, reading pages that are not cached.  1 = done, 0 = the kernel
// lacks MADV_POPULATE_READ (nothing done), -1 = a page could not be read.
int populate_range(const st_files_s &f, uint64_t begin, uint64_t end, std::string *msg) {
  static const uint64_t page = static_cast<uint64_t>(sysconf(_SC_PAGESIZE));
  for (const auto &p : f.parts) {
    const uint64_t a = std::max(begin, p.base), b = std::min(end, p.base + p.bytes);
    if (a >= b || !p.map) continue;
    const uint64_t lo = (p.offset + (a - p.base)) / page * page;
    const uint64_t hi = std::min(p.map_bytes, p.offset + (b - p.base));
    if (madvise(const_cast<uint8_t *>(p.map) + lo, hi - lo, MADV_POPULATE_READ) != 0) {
      if (errno == EINVAL) return 0;
      *msg = "reading bytes " + std::to_string(lo) + ".." + std::to_string(hi) + " of " + p.path + " (mapped): " +
             std::strerror(errno) + " (did the file shrink?)";
      return -1;
    }
  }
  return 1;
}

}  // namespace

// Populate threads: jobs of at most kJob arena bytes in arena order, taken by
// `threads` workers; the job list of chunk k is [first[k], first[k + 1]).
struct Populator {
  static constexpr uint64_t kJob = 32ull << 20;
  const st_files_s *files;
  std::vector<uint64_t> lo, hi;
  std::vector<size_t> first;
  std::vector<int8_t> state;  // 0 pending, 1 done, -1 failed (guarded by m)
  std::vector<std::string> msg;
  std::atomic<size_t> next{0};
  std::atomic<bool> stop{false};
  std::mutex m;
  std::condition_variable cv;
  std::vector<std::thread> pool;
};

Populator *populate_start(const st_files_s *f, uint64_t begin, uint64_t bytes, uint64_t chunk,
                          uint32_t threads) try {
  std::unique_ptr<Populator> own(new Populator);
  Populator *P = own.get();
  P->files = f;
  const uint64_t C = chunk ? chunk : (bytes ? bytes : 1), end = begin + bytes;
  for (uint64_t c0 = begin; c0 < end; c0 += C) {
    P->first.push_back(P->lo.size());
    const uint64_t c1 = std::min(end, c0 + C);
    for (uint64_t x = c0; x < c1; x += Populator::kJob) {
      P->lo.push_back(x);
      P->hi.push_back(std::min(c1, x + Populator::kJob));
    }
  }
  P->first.push_back(P->lo.size());
  P->state.assign(P->lo.size(), 0);
  P->msg.resize(P->lo.size());
  const uint32_t t = std::min<uint32_t>(threads, 16);  // 0: populate_wait does the jobs on the calling thread
  try {
    for (uint32_t i = 0; i < t && i < P->lo.size(); ++i)
      P->pool.emplace_back([P] {
        bool supported = true;
        for (;;) {
          const size_t j = P->next.fetch_add(1);
          if (j >= P->lo.size() || P->stop.load()) break;
          std::string msg;
          const int r = supported ? populate_range(*P->files, P->lo[j], P->hi[j], &msg) : 0;
          if (r == 0) supported = false;
          {
            std::lock_guard<std::mutex> g(P->m);
            P->state[j] = r < 0 ? -1 : 1;
            if (r < 0) P->msg[j] = std::move(msg);
          }
          P->cv.notify_all();
        }
      });
  } catch (const std::exception &) {
    // Fewer workers (or none): populate_wait then does the missing jobs itself.
  }
  return own.release();
} catch (const std::bad_alloc &) {
  return nullptr;
}

st_status populate_wait(Populator *P, uint64_t k) {
  if (k + 1 >= P->first.size()) return ST_OK;
  std::unique_lock<std::mutex> g(P->m);
  for (size_t j = P->first[k]; j < P->first[k + 1]; ++j) {
    if (P->pool.empty() && P->state[j] == 0) {  // no workers: populate here
      g.unlock();
      std::string msg;
      const int r = populate_range(*P->files, P->lo[j], P->hi[j], &msg);
      g.lock();
      P->state[j] = r < 0 ? -1 : 1;
      if (r < 0) P->msg[j] = std::move(msg);
    }
    P->cv.wait(g, [&] { return P->state[j] != 0; });
    if (P->state[j] < 0) return set_error(ST_E_IO, "%s", P->msg[j].c_str());
  }
  return ST_OK;
}

void populate_stop(Populator *P) {
  if (!P) return;
  P->stop = true;
  for (auto &th : P->pool) th.join();
  delete P;
}

st_status copy_arena_direct(const st_files_s *f, uint64_t begin, uint64_t bytes, void *dev, void *stream) {
  if (begin > f->arena_bytes || bytes > f->arena_bytes - begin)
    return set_error(ST_E_INVAL, "range %llu + %llu is beyond the %llu-byte arena", (unsigned long long)begin,
                     (unsigned long long)bytes, (unsigned long long)f->arena_bytes);
  for (const auto &p : f->parts) {
    const uint64_t a = std::max(begin, p.base), b = std::min(begin + bytes, p.base + p.bytes);
    if (a >= b) continue;
    if (!p.map) return set_error(ST_E_IO, "%s could not be mapped: pass a pinned ring instead", p.path.c_str());
    const cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t *>(dev) + (a - begin), p.map + p.offset + (a - p.base),
                                          b - a, cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
      return set_error(ST_E_CUDA, "copy of %llu bytes of %s: %s", (unsigned long long)(b - a), p.path.c_str(),
                       cudaGetErrorString(e));
  }
  return ST_OK;
}

}  // namespace stmat

using namespace stmat;

extern "C" {

st_status st_index_open(const char *path, st_index_t **out, uint64_t *data_offset) {
  if (!path || !out) return set_error(ST_E_INVAL, "NULL argument");
  *out = nullptr;
  const int fd = open(path, O_RDONLY | O_CLOEXEC);
  if (fd < 0) return set_error(ST_E_IO, "opening %s: %s", path, std::strerror(errno));
  struct FdGuard {
    int fd;
    ~FdGuard() { close(fd); }
  } guard{fd};
  struct stat sb;
  if (fstat(fd, &sb) != 0) return set_error(ST_E_IO, "stat %s: %s", path, std::strerror(errno));
  const uint64_t size = static_cast<uint64_t>(sb.st_size);
  uint8_t first[8];
  int err = 0;
  if (size < 8 || !pread_all(fd, first, 8, 0, &err))
    return set_error(ST_E_TRUNCATED, "%s holds %llu bytes, fewer than the 8-byte header length", path,
                     (unsigned long long)size);
  uint64_t n = 0;
  st_status s = st_header_size(first, 8, &n);
  if (s != ST_OK) return s;
  if (n > size - 8)
    return set_error(ST_E_TRUNCATED, "%s: header of %llu bytes but only %llu follow", path, (unsigned long long)n,
                     (unsigned long long)(size - 8));
  std::vector<uint8_t> hdr;
  try {
    hdr.resize(8 + n);
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory");
  }
  std::memcpy(hdr.data(), first, 8);
  if (n && !pread_all(fd, hdr.data() + 8, n, 8, &err))
    return set_error(ST_E_IO, "reading the header of %s: %s", path, err ? std::strerror(err) : "the file ended early");
  s = st_index_build(hdr.data(), hdr.size(), size - 8 - n, out);
  if (s == ST_OK && data_offset) *data_offset = 8 + n;
  return s;
}

st_status st_files_open(const st_file_part *parts, size_t n, st_files_t **out) {
  if (!out || (n && !parts)) return set_error(ST_E_INVAL, "NULL argument");
  *out = nullptr;
  static std::atomic<uint64_t> next_uid{1};
  std::unique_ptr<st_files_s> f(new (std::nothrow) st_files_s);
  if (!f) return set_error(ST_E_NOMEM, "out of host memory");
  f->uid = next_uid.fetch_add(1);
  try {
    for (size_t k = 0; k < n; ++k) {
      const st_file_part &p = parts[k];
      if (!p.path) return set_error(ST_E_INVAL, "NULL path of part %zu", k);
      if (p.base + p.bytes < p.base || p.offset + p.bytes < p.offset)
        return set_error(ST_E_INVAL, "part %zu overflows 64 bits", k);
      st_files_s::Part q;
      q.path = p.path;
      q.offset = p.offset;
      q.bytes = p.bytes;
      q.base = p.base;
      q.fd = open(p.path, O_RDONLY | O_CLOEXEC);
      if (q.fd < 0) return set_error(ST_E_IO, "opening %s: %s", p.path, std::strerror(errno));
      f->parts.push_back(std::move(q));
      struct stat sb;
      if (fstat(f->parts.back().fd, &sb) != 0) return set_error(ST_E_IO, "stat %s: %s", p.path, std::strerror(errno));
      if (static_cast<uint64_t>(sb.st_size) < p.offset + p.bytes)
        return set_error(ST_E_IO, "%s holds %llu bytes; part %zu needs %llu", p.path, (unsigned long long)sb.st_size,
                         k, (unsigned long long)(p.offset + p.bytes));
      if (sb.st_size > 0) {  // a failed mapping only rules out ring-less loads
        void *m = mmap(nullptr, static_cast<size_t>(sb.st_size), PROT_READ, MAP_SHARED, f->parts.back().fd, 0);
        if (m != MAP_FAILED) {
          f->parts.back().map = static_cast<const uint8_t *>(m);
          f->parts.back().map_bytes = static_cast<uint64_t>(sb.st_size);
        }
      }
    }
    std::sort(f->parts.begin(), f->parts.end(),
              [](const st_files_s::Part &a, const st_files_s::Part &b) { return a.base < b.base; });
    for (size_t k = 0; k < f->parts.size(); ++k) {
      const auto &p = f->parts[k];
      if (k && f->parts[k - 1].base + f->parts[k - 1].bytes > p.base)
        return set_error(ST_E_INVAL, "parts overlap in the arena at %llu", (unsigned long long)p.base);
      f->arena_bytes = std::max(f->arena_bytes, p.base + p.bytes);
    }
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory");
  }
  *out = f.release();
  return ST_OK;
}

void st_files_close(st_files_t *files) { delete files; }

st_status st_files_read(const st_files_t *files, uint64_t begin, uint64_t bytes, void *host, uint32_t threads) {
  return read_arena(files, begin, bytes, host, threads);
}

st_status st_files_prefetch(const st_files_t *files, uint64_t begin, uint64_t bytes, uint32_t threads) {
  if (!files) return set_error(ST_E_INVAL, "NULL files");
  if (begin > files->arena_bytes || bytes > files->arena_bytes - begin)
    return set_error(ST_E_INVAL, "range %llu + %llu is beyond the %llu-byte arena", (unsigned long long)begin,
                     (unsigned long long)bytes, (unsigned long long)files->arena_bytes);
  if (!bytes) return ST_OK;
  Populator *P = populate_start(files, begin, bytes, 0, threads);
  if (!P) return set_error(ST_E_NOMEM, "starting the populate threads");
  const st_status s = populate_wait(P, 0);
  populate_stop(P);
  return s;
}

st_status st_device_reads_pageable(int device, int32_t *yes) {
  if (!yes) return set_error(ST_E_INVAL, "NULL argument");
  int v = 0;
  const cudaError_t e = cudaDeviceGetAttribute(&v, cudaDevAttrPageableMemoryAccessUsesHostPageTables, device);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "device %d: %s", device, cudaGetErrorString(e));
  *yes = v ? 1 : 0;
  return ST_OK;
}

}  // extern "C"

// ------------------------------------------------------------ RAM tier
//
// "Disk tier integration": an LRU cache of host copies of tensors read from
// disk, bounded by a configurable number of bytes; evicting an entry drops
// the host copy (the tensor stays described by the index and is read again
// on its next use).  An entry is keyed by (files, arena range); get() holds
// it until release(), and held entries are never evicted.  An entry larger
// than the bound is read but not kept (dropped on release).

#include <list>
#include <map>
#include <mutex>
#include <tuple>

struct st_cache_s {
  struct Entry {
    uint64_t files;  // the files' uid
    uint64_t begin, bytes;
    uint8_t *host = nullptr;
    uint32_t holds = 0;
    bool kept = true;  // counted in `bytes` and listed in the LRU order
  };
  using Key = std::tuple<uint64_t, uint64_t, uint64_t>;  // (files uid, begin, bytes)
  uint64_t max_bytes = 0, bytes = 0, hits = 0, misses = 0, evictions = 0;
  bool pinned = false;
  std::mutex mu;
  std::list<Entry> lru;                                  // front = most recently used
  std::map<Key, std::list<Entry>::iterator> by_key;
  std::map<const void *, std::list<Entry>::iterator> by_ptr;
  std::list<Entry> transient;                            // too large to keep
  // Holds handed over by st_load_tensors: released once the event (recorded
  // after the copies that read those entries) has completed.
  struct Pending {
    cudaEvent_t ev;
    std::vector<const void *> hosts;
  };
  std::vector<Pending> pending;

  uint8_t *alloc(uint64_t n) {
    void *p = nullptr;
    if (pinned) {
      if (cudaHostAlloc(&p, n ? n : 1, cudaHostAllocDefault) != cudaSuccess) return nullptr;
    } else {
      p = std::malloc(n ? n : 1);
    }
    return static_cast<uint8_t *>(p);
  }
  void dealloc(uint8_t *p) {
    if (!p) return;
    if (pinned) cudaFreeHost(p);
    else std::free(p);
  }
  // Evicts least-recently-used unheld entries until `need` more bytes fit.
  void make_room(uint64_t need) {
    for (auto it = lru.end(); bytes + need > max_bytes && it != lru.begin();) {
      --it;
      if (it->holds) continue;
      bytes -= it->bytes;
      ++evictions;
      by_key.erase(Key(it->files, it->begin, it->bytes));
      by_ptr.erase(it->host);
      dealloc(it->host);
      it = lru.erase(it);
    }
  }
  // Drops one hold (mu held); an entry too large to keep is freed with its last hold.
  bool release_locked(const void *host) {
    auto it = by_ptr.find(host);
    if (it == by_ptr.end() || it->second->holds == 0) return false;
    auto e = it->second;
    if (--e->holds == 0 && !e->kept) {
      by_ptr.erase(it);
      dealloc(e->host);
      transient.erase(e);
    }
    return true;
  }
  // Releases the pending holds whose copies have finished (mu held); with
  // `wait`, waits for all of them first.
  void reap(bool wait) {
    size_t kept = 0;
    for (size_t i = 0; i < pending.size(); ++i) {
      Pending &p = pending[i];
      cudaError_t e = wait ? cudaEventSynchronize(p.ev) : cudaEventQuery(p.ev);
      if (e == cudaErrorNotReady) {
        (void)cudaGetLastError();  // not-ready is recorded as the last error: clear it
        if (kept != i) pending[kept] = std::move(p);  // never onto itself: that would empty `hosts`
        ++kept;
        continue;
      }
      // Done, or the context failed (then no copy reads the entries any more).
      for (const void *h : p.hosts) release_locked(h);
      cudaEventDestroy(p.ev);
    }
    pending.resize(kept);
  }
  ~st_cache_s() {
    reap(true);
    for (Entry &e : lru) dealloc(e.host);
    for (Entry &e : transient) dealloc(e.host);
  }
};

namespace stmat {

bool cache_release_after(st_cache_s *c, void *event, const std::vector<const void *> &hosts) {
  std::lock_guard<std::mutex> lock(c->mu);
  try {
    c->pending.push_back({static_cast<cudaEvent_t>(event), hosts});
  } catch (const std::bad_alloc &) {
    return false;
  }
  return true;
}

}  // namespace stmat

extern "C" {

st_status st_cache_create(uint64_t max_bytes, int32_t pinned, st_cache_t **out) {
  if (!out) return set_error(ST_E_INVAL, "NULL out");
  st_cache_s *c = new (std::nothrow) st_cache_s;
  if (!c) return set_error(ST_E_NOMEM, "out of host memory");
  c->max_bytes = max_bytes;
  c->pinned = pinned != 0;
  *out = c;
  return ST_OK;
}

void st_cache_free(st_cache_t *cache) { delete cache; }

st_status st_cache_get(st_cache_t *c, const st_files_t *files, uint64_t begin, uint64_t bytes, uint32_t threads,
                       const void **host) {
  if (!c || !files || !host) return set_error(ST_E_INVAL, "NULL argument");
  *host = nullptr;
  std::lock_guard<std::mutex> lock(c->mu);
  c->reap(false);
  const st_cache_s::Key key(files->uid, begin, bytes);
  auto hit = c->by_key.find(key);
  if (hit != c->by_key.end()) {
    ++c->hits;
    c->lru.splice(c->lru.begin(), c->lru, hit->second);  // most recent
    ++hit->second->holds;
    *host = hit->second->host;
    return ST_OK;
  }
  ++c->misses;
  st_cache_s::Entry e;
  e.files = files->uid;
  e.begin = begin;
  e.bytes = bytes;
  e.kept = bytes <= c->max_bytes;
  if (e.kept) c->make_room(bytes);
  e.host = c->alloc(bytes);
  if (!e.host) return set_error(ST_E_NOMEM, "allocating %llu bytes of %s host memory", (unsigned long long)bytes,
                                c->pinned ? "pinned" : "pageable");
  st_status s = read_arena(files, begin, bytes, e.host, threads);
  if (s != ST_OK) {
    c->dealloc(e.host);
    return s;
  }
  e.holds = 1;
  try {
    if (e.kept) {
      c->lru.push_front(e);
      c->by_key[key] = c->lru.begin();
      c->by_ptr[e.host] = c->lru.begin();
      c->bytes += bytes;
    } else {
      c->transient.push_front(e);
      c->by_ptr[e.host] = c->transient.begin();
    }
  } catch (const std::bad_alloc &) {
    c->dealloc(e.host);
    return set_error(ST_E_NOMEM, "out of host memory");
  }
  *host = e.host;
  return ST_OK;
}

st_status st_cache_release(st_cache_t *c, const void *host) {
  if (!c || !host) return set_error(ST_E_INVAL, "NULL argument");
  std::lock_guard<std::mutex> lock(c->mu);
  if (!c->release_locked(host)) return set_error(ST_E_INVAL, "%p is not a held cache entry", host);
  return ST_OK;
}

st_status st_cache_stats(const st_cache_t *c, st_cache_info *info) {
  if (!c || !info) return set_error(ST_E_INVAL, "NULL argument");
  std::lock_guard<std::mutex> lock(const_cast<st_cache_s *>(c)->mu);
  const_cast<st_cache_s *>(c)->reap(false);
  info->bytes = c->bytes;
  info->max_bytes = c->max_bytes;
  info->entries = c->lru.size();
  info->hits = c->hits;
  info->misses = c->misses;
  info->evictions = c->evictions;
  return ST_OK;
}

st_status st_cache_clear(st_cache_t *c) {
  if (!c) return set_error(ST_E_INVAL, "NULL cache");
  std::lock_guard<std::mutex> lock(c->mu);
  c->reap(true);
  const uint64_t keep = c->max_bytes;
  c->max_bytes = 0;
  c->make_room(0);
  c->max_bytes = keep;
  return ST_OK;
}

}  // extern "C"

// ------------------------------------------------------------ host locality
//
// Pinned staging memory and the threads that fill it belong on the CPU
// socket the GPU hangs off: page-locked pages are placed where the thread
// that allocates them runs, and copies from a remote socket's memory cross
// the CPU interconnect.

#include <sched.h>

#include <cctype>

#include <fstream>

extern "C" {

st_status st_host_affinity(int device, int32_t apply, char *cpulist, size_t len) {
  char bus[64] = {0};
  cudaError_t e = cudaDeviceGetPCIBusId(bus, sizeof bus, device);
  if (e != cudaSuccess)
    return set_error(ST_E_CUDA, "cudaDeviceGetPCIBusId(%d): %s", device, cudaGetErrorString(e));
  for (char *c = bus; *c; ++c) *c = static_cast<char>(std::tolower(static_cast<unsigned char>(*c)));
  std::string path = std::string("/sys/bus/pci/devices/") + bus + "/local_cpulist";
  std::ifstream f(path);
  std::string list;
  if (!f || !std::getline(f, list) || list.empty())
    return set_error(ST_E_IO, "cannot read %s", path.c_str());
  if (cpulist && len) {
    std::strncpy(cpulist, list.c_str(), len - 1);
    cpulist[len - 1] = 0;
  }
  if (!apply) return ST_OK;
  cpu_set_t set;
  CPU_ZERO(&set);
  size_t i = 0;
  int count = 0;
  while (i < list.size()) {  // "a-b,c,d-e"
    size_t j = list.find(',', i);
    if (j == std::string::npos) j = list.size();
    const std::string item = list.substr(i, j - i);
    const size_t dash = item.find('-');
    char *end = nullptr;
    const long lo = std::strtol(item.c_str(), &end, 10);
    const long hi = dash == std::string::npos ? lo : std::strtol(item.c_str() + dash + 1, &end, 10);
    if (lo < 0 || hi < lo || hi >= CPU_SETSIZE) return set_error(ST_E_INVAL, "cannot parse cpu list \"%s\"", list.c_str());
    for (long c = lo; c <= hi; ++c) {
      CPU_SET(static_cast<int>(c), &set);
      ++count;
    }
    i = j + 1;
  }
  if (!count) return set_error(ST_E_INVAL, "empty cpu list for device %d", device);
  if (sched_setaffinity(0, sizeof set, &set) != 0)
    return set_error(ST_E_IO, "sched_setaffinity: %s", std::strerror(errno));
  return ST_OK;
}

}  // extern "C"
