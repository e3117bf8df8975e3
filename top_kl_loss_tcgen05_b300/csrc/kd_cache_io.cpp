// kd_cache_io.cpp - the teacher top-K cache on disk.
//
// The method computes the teacher's top-K once, offline, and reuses it for
// every training run ("ทำให้ Knowledge Distillation มีประสิทธิภาพ..."
// (ai-thai.com), section "การทำ Distillation แบบ Offline"; "Multiverse
// Computing сократила видеопамять..." (iitog.ru), fourth paragraph). The
// pages name no file format; this one is the plainest that serves a
// training loader: fixed-size records, one per position, so any range of
// positions is one contiguous read.
//
//   offset 0   "KDTOPK01"        8-byte magic
//          8   uint32 version    1
//         12   uint32 header     64 (bytes before the first record)
//         16   int64  T          records; -1 while a writer holds the file
//         24   int64  V          vocabulary size (ids lie in [0, V))
//         32   int32  K          entries per record
//         36   uint32 flags      0
//         40   24 zero bytes
//         64   T records of 8 K bytes: K int32 ids, then K float32 logp
// Little-endian throughout. Host memory only; nothing here touches the GPU.
#include <cerrno>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include "../../include/kd.h"

struct kd_cache_file {
  int fd = -1;
  bool writer = false;
  int64_t T = 0, V = 0;
  int32_t K = 0;
};

namespace {

constexpr char kMagic[8] = {'K', 'D', 'T', 'O', 'P', 'K', '0', '1'};
constexpr uint32_t kVersion = 1;
constexpr uint32_t kHeaderBytes = 64;
constexpr size_t kIoBytes = size_t(8) << 20;  // staging buffer per read / append step

struct Header {
  char magic[8];
  uint32_t version;
  uint32_t header_bytes;
  int64_t T;
  int64_t V;
  int32_t K;
  uint32_t flags;
  uint8_t reserved[24];
};
static_assert(sizeof(Header) == kHeaderBytes, "header layout");

bool write_all(int fd, const void* p, size_t n, off_t off) {
  const char* c = static_cast<const char*>(p);
  while (n > 0) {
    const ssize_t w = pwrite(fd, c, n, off);
    if (w < 0 && errno == EINTR) continue;
    if (w <= 0) return false;
    c += w;
    n -= (size_t)w;
    off += w;
  }
  return true;
}

// Reads exactly n bytes; false on an error or a short file.
bool read_all(int fd, void* p, size_t n, off_t off) {
  char* c = static_cast<char*>(p);
  while (n > 0) {
    const ssize_t r = pread(fd, c, n, off);
    if (r < 0 && errno == EINTR) continue;
    if (r <= 0) return false;
    c += r;
    n -= (size_t)r;
    off += r;
  }
  return true;
}

size_t record_bytes(int32_t K) { return (size_t)K * 8; }

}  // namespace

extern "C" {

int kd_cache_create(const char* path, int64_t V, int32_t K, kd_cache_file** out) {
  if (!path || !out || V <= 0 || K <= 0 || K > V || V >= (int64_t(1) << 31)) return KD_ERR_INVALID_ARG;
  *out = nullptr;
  const int fd = open(path, O_WRONLY | O_CREAT | O_TRUNC | O_CLOEXEC, 0644);
  if (fd < 0) return KD_ERR_IO;
  Header h;
  std::memset(&h, 0, sizeof(h));
  std::memcpy(h.magic, kMagic, 8);
  h.version = kVersion;
  h.header_bytes = kHeaderBytes;
  h.T = -1;  // unfinished until kd_cache_close
  h.V = V;
  h.K = K;
  if (!write_all(fd, &h, sizeof(h), 0)) {
    close(fd);
    return KD_ERR_IO;
  }
  kd_cache_file* f = new (std::nothrow) kd_cache_file;
  if (!f) {
    close(fd);
    return KD_ERR_IO;
  }
  f->fd = fd;
  f->writer = true;
  f->T = 0;
  f->V = V;
  f->K = K;
  *out = f;
  return KD_OK;
}

int kd_cache_append(kd_cache_file* f, const int32_t* ids, const float* logp, int64_t rows) {
  if (!f || !f->writer || rows < 0) return KD_ERR_INVALID_ARG;
  if (rows == 0) return KD_OK;
  if (!ids || !logp) return KD_ERR_INVALID_ARG;
  const int32_t K = f->K;
  for (int64_t i = 0; i < rows * K; ++i)
    if (ids[i] < 0 || ids[i] >= f->V) return KD_ERR_BAD_ID;  // nothing written
  const size_t rb = record_bytes(K);
  const int64_t per = (int64_t)(kIoBytes / rb > 0 ? kIoBytes / rb : 1);
  std::vector<char> buf;
  try {
    buf.resize((size_t)(rows < per ? rows : per) * rb);
  } catch (...) {
    return KD_ERR_IO;
  }
  for (int64_t r0 = 0; r0 < rows; r0 += per) {
    const int64_t n = (rows - r0) < per ? (rows - r0) : per;
    for (int64_t r = 0; r < n; ++r) {
      char* rec = buf.data() + (size_t)r * rb;
      std::memcpy(rec, ids + (r0 + r) * K, (size_t)K * 4);
      std::memcpy(rec + (size_t)K * 4, logp + (r0 + r) * K, (size_t)K * 4);
    }
    const off_t off = (off_t)kHeaderBytes + (off_t)(f->T + r0) * (off_t)rb;
    if (!write_all(f->fd, buf.data(), (size_t)n * rb, off)) return KD_ERR_IO;
  }
  f->T += rows;
  return KD_OK;
}

int kd_cache_open(const char* path, kd_cache_file** out, int64_t* T, int64_t* V, int32_t* K) {
  if (!path || !out) return KD_ERR_INVALID_ARG;
  *out = nullptr;
  const int fd = open(path, O_RDONLY | O_CLOEXEC);
  if (fd < 0) return KD_ERR_IO;
  Header h;
  struct stat st;
  int rc = KD_OK;
  if (fstat(fd, &st) != 0) rc = KD_ERR_IO;
  else if (!read_all(fd, &h, sizeof(h), 0)) rc = KD_ERR_FORMAT;
  else if (std::memcmp(h.magic, kMagic, 8) != 0 || h.version != kVersion || h.header_bytes != kHeaderBytes)
    rc = KD_ERR_FORMAT;
  else if (h.T < 0 || h.V <= 0 || h.K <= 0 || h.K > h.V || h.V >= (int64_t(1) << 31))
    rc = KD_ERR_FORMAT;  // unfinished (writer never closed) or corrupt
  else if ((uint64_t)st.st_size != (uint64_t)kHeaderBytes + (uint64_t)h.T * record_bytes(h.K))
    rc = KD_ERR_FORMAT;  // truncated or trailing bytes
  if (rc != KD_OK) {
    close(fd);
    return rc;
  }
  kd_cache_file* f = new (std::nothrow) kd_cache_file;
  if (!f) {
    close(fd);
    return KD_ERR_IO;
  }
  f->fd = fd;
  f->writer = false;
  f->T = h.T;
  f->V = h.V;
  f->K = h.K;
  if (T) *T = h.T;
  if (V) *V = h.V;
  if (K) *K = h.K;
  *out = f;
  return KD_OK;
}

int kd_cache_read(kd_cache_file* f, int64_t row0, int64_t rows, int32_t* ids, float* logp) {
  if (!f || f->writer || row0 < 0 || rows < 0 || row0 + rows > f->T) return KD_ERR_INVALID_ARG;
  if (rows == 0) return KD_OK;
  if (!ids || !logp) return KD_ERR_INVALID_ARG;
  const int32_t K = f->K;
  const size_t rb = record_bytes(K);
  const int64_t per = (int64_t)(kIoBytes / rb > 0 ? kIoBytes / rb : 1);
  std::vector<char> buf;
  try {
    buf.resize((size_t)(rows < per ? rows : per) * rb);
  } catch (...) {
    return KD_ERR_IO;
  }
  for (int64_t r0 = 0; r0 < rows; r0 += per) {
    const int64_t n = (rows - r0) < per ? (rows - r0) : per;
    const off_t off = (off_t)kHeaderBytes + (off_t)(row0 + r0) * (off_t)rb;
    if (!read_all(f->fd, buf.data(), (size_t)n * rb, off)) return KD_ERR_IO;
    for (int64_t r = 0; r < n; ++r) {
      const char* rec = buf.data() + (size_t)r * rb;
      std::memcpy(ids + (r0 + r) * K, rec, (size_t)K * 4);
      std::memcpy(logp + (r0 + r) * K, rec + (size_t)K * 4, (size_t)K * 4);
    }
  }
  return KD_OK;
}

int kd_cache_close(kd_cache_file* f) {
  if (!f) return KD_ERR_INVALID_ARG;
  int rc = KD_OK;
  if (f->writer) {
    // Record the row count last: a file whose writer never got here keeps
    // T = -1 and is rejected by kd_cache_open.
    const int64_t T = f->T;
    if (fdatasync(f->fd) != 0 || !write_all(f->fd, &T, sizeof(T), 16) || fdatasync(f->fd) != 0) rc = KD_ERR_IO;
  }
  if (close(f->fd) != 0 && rc == KD_OK) rc = KD_ERR_IO;
  delete f;
  return rc;
}

}  // extern "C"
