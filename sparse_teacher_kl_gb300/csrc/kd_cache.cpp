// On-disk teacher top-K cache: write once after the teacher's single pass, read
// back in row ranges for every training run ([ART] paragraph on the first fix:
// the teacher runs once, its top-K logits per position are stored on disk and
// reused across experiments; [DAI] "As duas inovações" item 1).
//
// One file ("shard") per contiguous range of positions.  Layout, little-endian:
//   header (64 bytes)
//     0  char[8]  magic "KDTOPK\0\1"
//     8  u32      format version (1)
//     12 u32      K
//     16 u64      V (vocabulary size of the teacher)
//     24 u64      N (positions in this shard)
//     32 u64      row0 (global index of the shard's first position)
//     40 u32      logits type: 0 = fp32, 1 = bf16
//     44 u32      flags: bit 0 = a per-position teacher logsumexp follows
//     48 u64      FNV-1a 64 of the payload
//     56 u64      reserved (0)
//   payload
//     ids     int32 [N, K]
//     logits  fp32 or bf16 [N, K]
//     lse     fp32 [N]            (if flags bit 0)
// bf16 storage halves the logits on disk; it is exact for caches extracted from
// bf16 teacher logits (every value is a widened bf16).  Host code only.
#include <errno.h>
#include <algorithm>
#include <fcntl.h>
#include <stdio.h>
#include <string.h>
#include <sys/stat.h>
#include <unistd.h>

#include <condition_variable>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "../../include/kdkl.h"

namespace {

constexpr char kMagic[8] = {'K', 'D', 'T', 'O', 'P', 'K', '\0', '\1'};
constexpr uint32_t kVersion = 1;

struct Header {
  char magic[8];
  uint32_t version;
  uint32_t K;
  uint64_t V;
  uint64_t N;
  uint64_t row0;
  uint32_t logits_type;
  uint32_t flags;
  uint64_t checksum;
  uint64_t reserved;
};
static_assert(sizeof(Header) == 64, "cache header is 64 bytes");

struct Fnv {
  uint64_t h = 1469598103934665603ull;
  void add(const void* p, size_t n) {
    const uint8_t* b = static_cast<const uint8_t*>(p);
    for (size_t i = 0; i < n; ++i) {
      h ^= b[i];
      h *= 1099511628211ull;
    }
  }
};

bool write_all(int fd, const void* p, size_t n) {
  const uint8_t* b = static_cast<const uint8_t*>(p);
  while (n > 0) {
    const ssize_t w = ::write(fd, b, n);
    if (w < 0) {
      if (errno == EINTR) continue;
      return false;
    }
    b += w;
    n -= size_t(w);
  }
  return true;
}

bool pread_all(int fd, void* p, size_t n, uint64_t off) {
  uint8_t* b = static_cast<uint8_t*>(p);
  while (n > 0) {
    const ssize_t r = ::pread(fd, b, n, off_t(off));
    if (r < 0) {
      if (errno == EINTR) continue;
      return false;
    }
    if (r == 0) return false;  // truncated
    b += r;
    n -= size_t(r);
    off += uint64_t(r);
  }
  return true;
}

// fp32 -> bf16 with round-to-nearest-even (NaN kept quiet).
uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return uint16_t((u >> 16) | 0x40u);
  const uint32_t round = 0x7fffu + ((u >> 16) & 1u);
  return uint16_t((u + round) >> 16);
}

float from_bf16(uint16_t b) {
  const uint32_t u = uint32_t(b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

int read_header(int fd, Header* h) {
  if (!pread_all(fd, h, sizeof(Header), 0)) return KD_ERR_IO;
  if (memcmp(h->magic, kMagic, 8) != 0 || h->version != kVersion) return KD_ERR_UNSUPPORTED;
  if (h->K < 1 || h->K > KD_MAX_K || h->V < h->K || h->logits_type > 1) return KD_ERR_UNSUPPORTED;
  return KD_OK;
}

uint64_t payload_bytes(const Header& h) {
  const uint64_t nk = h.N * uint64_t(h.K);
  return nk * 4 + nk * (h.logits_type == 1 ? 2 : 4) + ((h.flags & 1u) ? h.N * 4 : 0);
}

}  // namespace

extern "C" {

int kd_cache_write(const char* path, const int32_t* ids, const float* logits, const float* lse, int64_t N, int K,
                   int64_t V, int64_t row0, int logits_bf16) {
  if (!path || (N > 0 && (!ids || !logits)) || N < 0 || K < 1 || K > KD_MAX_K || V < K || row0 < 0)
    return KD_ERR_INVALID_ARG;
  Header h{};
  memcpy(h.magic, kMagic, 8);
  h.version = kVersion;
  h.K = uint32_t(K);
  h.V = uint64_t(V);
  h.N = uint64_t(N);
  h.row0 = uint64_t(row0);
  h.logits_type = logits_bf16 ? 1u : 0u;
  h.flags = lse ? 1u : 0u;

  const size_t nk = size_t(N) * size_t(K);
  std::vector<uint16_t> lb;
  if (logits_bf16) {
    lb.resize(nk);
    for (size_t i = 0; i < nk; ++i) lb[i] = to_bf16(logits[i]);
  }
  Fnv fnv;
  fnv.add(ids, nk * 4);
  if (logits_bf16) fnv.add(lb.data(), nk * 2); else fnv.add(logits, nk * 4);
  if (lse) fnv.add(lse, size_t(N) * 4);
  h.checksum = fnv.h;

  const std::string tmp = std::string(path) + ".tmp";
  const int fd = ::open(tmp.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
  if (fd < 0) return KD_ERR_IO;
  bool ok = write_all(fd, &h, sizeof(h)) && write_all(fd, ids, nk * 4);
  ok = ok && (logits_bf16 ? write_all(fd, lb.data(), nk * 2) : write_all(fd, logits, nk * 4));
  if (lse) ok = ok && write_all(fd, lse, size_t(N) * 4);
  ok = (::fsync(fd) == 0) && ok;
  ok = (::close(fd) == 0) && ok;
  if (!ok || ::rename(tmp.c_str(), path) != 0) {
    ::unlink(tmp.c_str());
    return KD_ERR_IO;
  }
  return KD_OK;
}

int kd_cache_info(const char* path, int64_t* N, int* K, int64_t* V, int64_t* row0, int* logits_bf16, int* has_lse) {
  if (!path) return KD_ERR_INVALID_ARG;
  const int fd = ::open(path, O_RDONLY);
  if (fd < 0) return KD_ERR_IO;
  Header h{};
  int st = read_header(fd, &h);
  if (st == KD_OK) {
    struct stat sb;
    if (::fstat(fd, &sb) != 0 || uint64_t(sb.st_size) != sizeof(Header) + payload_bytes(h)) st = KD_ERR_IO;
  }
  ::close(fd);
  if (st != KD_OK) return st;
  if (N) *N = int64_t(h.N);
  if (K) *K = int(h.K);
  if (V) *V = int64_t(h.V);
  if (row0) *row0 = int64_t(h.row0);
  if (logits_bf16) *logits_bf16 = int(h.logits_type);
  if (has_lse) *has_lse = int(h.flags & 1u);
  return KD_OK;
}

int kd_cache_verify(const char* path) {
  if (!path) return KD_ERR_INVALID_ARG;
  const int fd = ::open(path, O_RDONLY);
  if (fd < 0) return KD_ERR_IO;
  Header h{};
  int st = read_header(fd, &h);
  if (st == KD_OK) {
    Fnv fnv;
    std::vector<uint8_t> buf(1 << 20);
    uint64_t left = payload_bytes(h), off = sizeof(Header);
    while (left > 0 && st == KD_OK) {
      const size_t n = size_t(left < buf.size() ? left : buf.size());
      if (!pread_all(fd, buf.data(), n, off)) st = KD_ERR_IO;
      fnv.add(buf.data(), n);
      left -= n;
      off += n;
    }
    if (st == KD_OK && fnv.h != h.checksum) st = KD_ERR_IO;
    uint8_t extra;
    if (st == KD_OK && ::pread(fd, &extra, 1, off_t(off)) != 0) st = KD_ERR_IO;
  }
  ::close(fd);
  return st;
}

int kd_cache_read(const char* path, int64_t first, int64_t count, int32_t* ids_out, float* logits_out,
                  float* lse_out) {
  if (!path || first < 0 || count < 0 || (count > 0 && (!ids_out || !logits_out))) return KD_ERR_INVALID_ARG;
  const int fd = ::open(path, O_RDONLY);
  if (fd < 0) return KD_ERR_IO;
  Header h{};
  int st = read_header(fd, &h);
  if (st == KD_OK && uint64_t(first + count) > h.N) st = KD_ERR_INVALID_ARG;
  if (st == KD_OK && lse_out && !(h.flags & 1u)) st = KD_ERR_INVALID_ARG;
  if (st == KD_OK && count > 0) {
    const uint64_t K = h.K, nk = h.N * K;
    const uint64_t ids_off = sizeof(Header);
    const uint64_t log_off = ids_off + nk * 4;
    const uint64_t lse_off = log_off + nk * (h.logits_type == 1 ? 2 : 4);
    const size_t n = size_t(count) * size_t(K);
    bool ok = pread_all(fd, ids_out, n * 4, ids_off + uint64_t(first) * K * 4);
    if (ok && h.logits_type == 1) {
      std::vector<uint16_t> lb(n);
      ok = pread_all(fd, lb.data(), n * 2, log_off + uint64_t(first) * K * 2);
      for (size_t i = 0; ok && i < n; ++i) logits_out[i] = from_bf16(lb[i]);
    } else if (ok) {
      ok = pread_all(fd, logits_out, n * 4, log_off + uint64_t(first) * K * 4);
    }
    if (ok && lse_out) ok = pread_all(fd, lse_out, size_t(count) * 4, lse_off + uint64_t(first) * 4);
    if (!ok) st = KD_ERR_IO;
  }
  ::close(fd);
  return st;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Streaming reader: batches of consecutive positions, the next batch read from
// disk on a background thread while the caller works on the current one.

namespace {

struct Reader {
  int fd = -1;
  Header h{};
  int64_t batch = 0;
  int64_t next_row = 0;  // first row of the batch being / to be prefetched
  std::vector<int32_t> ids;
  std::vector<float> logits;
  int64_t rows_ready = -1;  // rows in the prefetched batch, -1 = not ready
  int status = KD_OK;
  bool stop = false;
  bool want = true;  // a prefetch is requested
  std::mutex mu;
  std::condition_variable cv;
  std::thread worker;

  void run() {
    std::unique_lock<std::mutex> lock(mu);
    while (true) {
      cv.wait(lock, [&] { return stop || want; });
      if (stop) return;
      want = false;
      const int64_t first = next_row;
      const int64_t n = first < int64_t(h.N) ? std::min<int64_t>(batch, int64_t(h.N) - first) : 0;
      lock.unlock();
      int st = KD_OK;
      if (n > 0) st = read_rows(first, n);
      lock.lock();
      status = st;
      rows_ready = n;
      cv.notify_all();
    }
  }

  int read_rows(int64_t first, int64_t n) {
    const uint64_t K = h.K, nk = h.N * K;
    const uint64_t log_off = sizeof(Header) + nk * 4;
    const size_t cnt = size_t(n) * size_t(K);
    if (!pread_all(fd, ids.data(), cnt * 4, sizeof(Header) + uint64_t(first) * K * 4)) return KD_ERR_IO;
    if (h.logits_type == 1) {
      std::vector<uint16_t> lb(cnt);
      if (!pread_all(fd, lb.data(), cnt * 2, log_off + uint64_t(first) * K * 2)) return KD_ERR_IO;
      for (size_t i = 0; i < cnt; ++i) logits[i] = from_bf16(lb[i]);
    } else if (!pread_all(fd, logits.data(), cnt * 4, log_off + uint64_t(first) * K * 4)) {
      return KD_ERR_IO;
    }
    return KD_OK;
  }
};

}  // namespace

extern "C" {

int kd_cache_reader_open(const char* path, int64_t rows_per_batch, void** handle) {
  if (!path || rows_per_batch < 1 || !handle) return KD_ERR_INVALID_ARG;
  *handle = nullptr;
  Reader* r = new Reader();
  r->fd = ::open(path, O_RDONLY);
  if (r->fd < 0) {
    delete r;
    return KD_ERR_IO;
  }
  const int st = read_header(r->fd, &r->h);
  if (st != KD_OK) {
    ::close(r->fd);
    delete r;
    return st;
  }
  r->batch = rows_per_batch;
  r->ids.resize(size_t(rows_per_batch) * r->h.K);
  r->logits.resize(size_t(rows_per_batch) * r->h.K);
  r->worker = std::thread([r] { r->run(); });
  *handle = r;
  return KD_OK;
}

int kd_cache_reader_next(void* handle, int32_t* ids_out, float* logits_out, int64_t* rows_out) {
  if (!handle || !ids_out || !logits_out || !rows_out) return KD_ERR_INVALID_ARG;
  Reader* r = static_cast<Reader*>(handle);
  std::unique_lock<std::mutex> lock(r->mu);
  r->cv.wait(lock, [&] { return r->rows_ready >= 0; });
  const int st = r->status;
  const int64_t n = r->rows_ready;
  if (st == KD_OK && n > 0) {
    memcpy(ids_out, r->ids.data(), size_t(n) * r->h.K * 4);
    memcpy(logits_out, r->logits.data(), size_t(n) * r->h.K * 4);
  }
  *rows_out = st == KD_OK ? n : 0;
  if (st == KD_OK && n > 0) {
    r->next_row += n;
    r->rows_ready = -1;
    r->want = true;
    r->cv.notify_all();
  }
  return st;
}

int kd_cache_reader_close(void* handle) {
  if (!handle) return KD_ERR_INVALID_ARG;
  Reader* r = static_cast<Reader*>(handle);
  {
    std::lock_guard<std::mutex> lock(r->mu);
    r->stop = true;
  }
  r->cv.notify_all();
  r->worker.join();
  ::close(r->fd);
  delete r;
  return KD_OK;
}

}  // extern "C"
