// Shard-on-read from a safetensors file (include/tp_safetensors.h).
//
// diffusers "Tensor parallelism" page, §Load a sharded model: every rank reads
// only its slice of each weight and places it straight on its device.  The
// header is parsed once; each load moves the bytes of the requested ranks'
// slices in windows of the staging size, through one of two slot pairs:
//   staged: two page-locked staging buffers; while the copy engine moves one
//           buffer to the device, host threads read the next part of the file
//           into the other;
//   mapped: where the GPU reads pageable memory through the host's page
//           tables, the copy engine reads straight from a read-only mapping
//           of the file; the pages of each range are populated first, so the
//           copy finds them mapped (a copy that has to fault them in through
//           the GPU's address translation runs at about half the rate) and a
//           read error is reported instead of faulted on.  Pages stay mapped
//           until the file is closed: unmapping them after each copy costs
//           the TLB invalidations of every page, about as long as the copy.
// Colwise slices are contiguous row ranges of the file and are copied as they
// are; rowwise slices are scattered column segments, so whole rows are moved
// (to the pinned staging buffer, or to a device staging buffer when mapped)
// and the ranks' columns extracted by tp_plan_shard_ranks.
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <condition_variable>
#include <future>
#include <memory>
#include <mutex>
#include <cerrno>
#include <cstdio>
#include <cstring>
#include <string>
#include <system_error>
#include <thread>
#include <unordered_map>
#include <vector>

#include "tp_internal.h"
#include "tp_safetensors.h"

#ifndef MADV_POPULATE_READ
#define MADV_POPULATE_READ 22  // Linux 5.14 and later
#endif

namespace tp {
namespace stf {

constexpr uint64_t kMaxHeaderBytes = 100000000ull;  // the format's own header-size limit
constexpr int kMaxJsonDepth = 64;

struct Entry {
  std::string name;
  tp_st_dtype dtype = TP_ST_U8;
  int ndim = 0;
  int64_t shape[TP_ST_MAX_DIMS] = {0};
  uint64_t begin = 0, end = 0;  // relative to the first data byte
};

struct DtypeName {
  const char* name;
  tp_st_dtype dtype;
  size_t size;
};

constexpr DtypeName kDtypes[] = {
    {"BOOL", TP_ST_BOOL, 1}, {"U8", TP_ST_U8, 1},   {"I8", TP_ST_I8, 1},       {"F8_E4M3", TP_ST_F8_E4M3, 1},
    {"F8_E5M2", TP_ST_F8_E5M2, 1}, {"I16", TP_ST_I16, 2}, {"U16", TP_ST_U16, 2}, {"F16", TP_ST_F16, 2},
    {"BF16", TP_ST_BF16, 2}, {"I32", TP_ST_I32, 4}, {"U32", TP_ST_U32, 4},     {"F32", TP_ST_F32, 4},
    {"I64", TP_ST_I64, 8},   {"U64", TP_ST_U64, 8}, {"F64", TP_ST_F64, 8},
};

size_t dtype_size(tp_st_dtype d) {
  for (const auto& e : kDtypes)
    if (e.dtype == d) return e.size;
  return 0;
}

// A small JSON reader for the header: strings with every escape, integers for
// shapes and offsets, and any other value skipped over (bounded nesting).
class Json {
 public:
  explicit Json(const std::string& text) : s_(text) {}

  bool fail(const char* what) {
    if (err_.empty()) err_ = std::string(what) + " at header byte " + std::to_string(pos_);
    return false;
  }
  const std::string& error() const { return err_; }

  void ws() {
    while (pos_ < s_.size() && (s_[pos_] == ' ' || s_[pos_] == '\t' || s_[pos_] == '\n' || s_[pos_] == '\r')) ++pos_;
  }
  bool peek(char c) {
    ws();
    return pos_ < s_.size() && s_[pos_] == c;
  }
  bool expect(char c) {
    ws();
    if (pos_ >= s_.size() || s_[pos_] != c) {
      char msg[32];
      snprintf(msg, sizeof(msg), "expected '%c'", c);
      return fail(msg);
    }
    ++pos_;
    return true;
  }
  bool at_end() {
    ws();
    return pos_ == s_.size();
  }

  static void put_utf8(std::string& out, uint32_t cp) {
    if (cp < 0x80) {
      out += static_cast<char>(cp);
    } else if (cp < 0x800) {
      out += static_cast<char>(0xC0 | (cp >> 6));
      out += static_cast<char>(0x80 | (cp & 0x3F));
    } else if (cp < 0x10000) {
      out += static_cast<char>(0xE0 | (cp >> 12));
      out += static_cast<char>(0x80 | ((cp >> 6) & 0x3F));
      out += static_cast<char>(0x80 | (cp & 0x3F));
    } else {
      out += static_cast<char>(0xF0 | (cp >> 18));
      out += static_cast<char>(0x80 | ((cp >> 12) & 0x3F));
      out += static_cast<char>(0x80 | ((cp >> 6) & 0x3F));
      out += static_cast<char>(0x80 | (cp & 0x3F));
    }
  }

  bool hex4(uint32_t* v) {
    if (pos_ + 4 > s_.size()) return fail("truncated \\u escape");
    uint32_t x = 0;
    for (int i = 0; i < 4; ++i) {
      const char c = s_[pos_++];
      x <<= 4;
      if (c >= '0' && c <= '9') x |= static_cast<uint32_t>(c - '0');
      else if (c >= 'a' && c <= 'f') x |= static_cast<uint32_t>(c - 'a' + 10);
      else if (c >= 'A' && c <= 'F') x |= static_cast<uint32_t>(c - 'A' + 10);
      else return fail("bad hex digit in \\u escape");
    }
    *v = x;
    return true;
  }

  bool string(std::string* out) {
    if (!expect('"')) return false;
    out->clear();
    while (true) {
      if (pos_ >= s_.size()) return fail("unterminated string");
      const char c = s_[pos_++];
      if (c == '"') return true;
      if (static_cast<unsigned char>(c) < 0x20) return fail("control character in string");
      if (c != '\\') {
        *out += c;
        continue;
      }
      if (pos_ >= s_.size()) return fail("unterminated escape");
      const char e = s_[pos_++];
      switch (e) {
        case '"': *out += '"'; break;
        case '\\': *out += '\\'; break;
        case '/': *out += '/'; break;
        case 'b': *out += '\b'; break;
        case 'f': *out += '\f'; break;
        case 'n': *out += '\n'; break;
        case 'r': *out += '\r'; break;
        case 't': *out += '\t'; break;
        case 'u': {
          uint32_t cp = 0;
          if (!hex4(&cp)) return false;
          if (cp >= 0xD800 && cp < 0xDC00) {  // high surrogate: a low one must follow
            uint32_t lo = 0;
            if (pos_ + 2 > s_.size() || s_[pos_] != '\\' || s_[pos_ + 1] != 'u') return fail("lone surrogate");
            pos_ += 2;
            if (!hex4(&lo)) return false;
            if (lo < 0xDC00 || lo >= 0xE000) return fail("bad surrogate pair");
            cp = 0x10000 + ((cp - 0xD800) << 10) + (lo - 0xDC00);
          } else if (cp >= 0xDC00 && cp < 0xE000) {
            return fail("lone surrogate");
          }
          put_utf8(*out, cp);
          break;
        }
        default: return fail("bad escape");
      }
    }
  }

  // A non-negative integer with no sign, fraction or exponent, below 2^63.
  bool read_uint(uint64_t* v) {
    ws();
    const size_t start = pos_;
    uint64_t x = 0;
    while (pos_ < s_.size() && s_[pos_] >= '0' && s_[pos_] <= '9') {
      const uint64_t d = static_cast<uint64_t>(s_[pos_] - '0');
      if (x > (static_cast<uint64_t>(INT64_MAX) - d) / 10) return fail("integer too large");
      x = x * 10 + d;
      ++pos_;
    }
    if (pos_ == start) return fail("expected a non-negative integer");
    if (pos_ < s_.size() && (s_[pos_] == '.' || s_[pos_] == 'e' || s_[pos_] == 'E'))
      return fail("expected an integer, found a fraction or exponent");
    if (pos_ - start > 1 && s_[start] == '0') return fail("leading zero in integer");
    *v = x;
    return true;
  }

  bool literal(const char* word) {
    const size_t n = strlen(word);
    if (s_.compare(pos_, n, word) != 0) return fail("bad literal");
    pos_ += n;
    return true;
  }

  bool skip_value(int depth = 0) {
    if (depth > kMaxJsonDepth) return fail("nesting too deep");
    ws();
    if (pos_ >= s_.size()) return fail("expected a value");
    const char c = s_[pos_];
    if (c == '"') {
      std::string tmp;
      return string(&tmp);
    }
    if (c == '{') {
      ++pos_;
      if (peek('}')) return expect('}');
      while (true) {
        std::string k;
        if (!string(&k) || !expect(':') || !skip_value(depth + 1)) return false;
        if (peek(',')) {
          ++pos_;
          continue;
        }
        return expect('}');
      }
    }
    if (c == '[') {
      ++pos_;
      if (peek(']')) return expect(']');
      while (true) {
        if (!skip_value(depth + 1)) return false;
        if (peek(',')) {
          ++pos_;
          continue;
        }
        return expect(']');
      }
    }
    if (c == 't') return literal("true");
    if (c == 'f') return literal("false");
    if (c == 'n') return literal("null");
    if (c == '-' || (c >= '0' && c <= '9')) {  // any JSON number
      if (c == '-') ++pos_;
      const size_t digits = pos_;
      while (pos_ < s_.size() && s_[pos_] >= '0' && s_[pos_] <= '9') ++pos_;
      if (pos_ == digits) return fail("bad number");
      if (pos_ < s_.size() && s_[pos_] == '.') {
        ++pos_;
        const size_t f = pos_;
        while (pos_ < s_.size() && s_[pos_] >= '0' && s_[pos_] <= '9') ++pos_;
        if (pos_ == f) return fail("bad number");
      }
      if (pos_ < s_.size() && (s_[pos_] == 'e' || s_[pos_] == 'E')) {
        ++pos_;
        if (pos_ < s_.size() && (s_[pos_] == '+' || s_[pos_] == '-')) ++pos_;
        const size_t x = pos_;
        while (pos_ < s_.size() && s_[pos_] >= '0' && s_[pos_] <= '9') ++pos_;
        if (pos_ == x) return fail("bad number");
      }
      return true;
    }
    return fail("unexpected character");
  }

  // One tensor's entry: {"dtype": ..., "shape": [...], "data_offsets": [b, e]}.
  bool tensor(Entry* t) {
    if (!expect('{')) return false;
    bool has_dtype = false, has_shape = false, has_offsets = false;
    if (peek('}')) return fail("empty tensor entry");
    while (true) {
      std::string key;
      if (!string(&key) || !expect(':')) return false;
      if (key == "dtype") {
        std::string d;
        if (!string(&d)) return false;
        bool known = false;
        for (const auto& e : kDtypes)
          if (d == e.name) {
            t->dtype = e.dtype;
            known = true;
          }
        if (!known) return fail(("unknown dtype \"" + d + "\"").c_str());
        has_dtype = true;
      } else if (key == "shape") {
        if (!expect('[')) return false;
        t->ndim = 0;
        if (!peek(']')) {
          while (true) {
            uint64_t v = 0;
            if (!read_uint(&v)) return false;
            if (t->ndim == TP_ST_MAX_DIMS) return fail("shape has too many dimensions");
            t->shape[t->ndim++] = static_cast<int64_t>(v);
            if (peek(',')) {
              ++pos_;
              continue;
            }
            break;
          }
        }
        if (!expect(']')) return false;
        has_shape = true;
      } else if (key == "data_offsets") {
        uint64_t b = 0, e = 0;
        if (!expect('[') || !read_uint(&b) || !expect(',') || !read_uint(&e) || !expect(']')) return false;
        t->begin = b;
        t->end = e;
        has_offsets = true;
      } else {
        if (!skip_value(1)) return false;
      }
      if (peek(',')) {
        ++pos_;
        continue;
      }
      if (!expect('}')) return false;
      break;
    }
    if (!has_dtype || !has_shape || !has_offsets) return fail("tensor entry lacks dtype, shape or data_offsets");
    return true;
  }

 private:
  const std::string& s_;
  size_t pos_ = 0;
  std::string err_;
};

// pread until `len` bytes are in, or fail.
bool read_exact(int fd, void* dst, uint64_t len, uint64_t off, std::string* err) {
  uint8_t* p = static_cast<uint8_t*>(dst);
  while (len > 0) {
    const size_t want = static_cast<size_t>(std::min<uint64_t>(len, 1ull << 30));
    const ssize_t got = pread(fd, p, want, static_cast<off_t>(off));
    if (got < 0) {
      if (errno == EINTR) continue;
      *err = std::string("read failed: ") + strerror(errno);
      return false;
    }
    if (got == 0) {
      *err = "file ended early";
      return false;
    }
    p += got;
    off += static_cast<uint64_t>(got);
    len -= static_cast<uint64_t>(got);
  }
  return true;
}

// One part of a staged read: `len` bytes at file offset `off` go to staging offset `at`.
struct Range {
  uint64_t off, len, at;
};

// A fixed pool of reader threads.  A job is a list of ranges; its bytes are split
// evenly over the pool (the calling thread takes the first share), whatever the
// range boundaries, so a staging buffer filled from several slices is read at the
// full parallel rate.
class ReadPool {
 public:
  // Starts up to threads - 1 workers (the caller is the first reader); if the system refuses a
  // thread, the pool runs with the workers it got.
  explicit ReadPool(int threads) {
    const int want = std::max(1, threads);
    for (int i = 1; i < want; ++i) {
      try {
        workers_.emplace_back([this, i] { loop(i); });
      } catch (const std::system_error&) {
        break;
      }
    }
    n_ = 1 + static_cast<int>(workers_.size());
  }
  ~ReadPool() {
    {
      std::lock_guard<std::mutex> lk(m_);
      stop_ = true;
    }
    cv_job_.notify_all();
    for (auto& t : workers_) t.join();
  }

  bool run(int fd, uint8_t* dst, const std::vector<Range>& ranges, std::string* err) {
    uint64_t total = 0;
    for (const auto& r : ranges) total += r.len;
    constexpr uint64_t kMinShare = 1ull << 20;
    const int parts = static_cast<int>(std::max<uint64_t>(1, std::min<uint64_t>(n_, total / kMinShare)));
    if (parts == 1) return read_share(fd, dst, ranges, 0, total, err);
    {
      std::lock_guard<std::mutex> lk(m_);
      fd_ = fd;
      dst_ = dst;
      ranges_ = &ranges;
      total_ = total;
      parts_ = parts;
      errs_.assign(n_, std::string());
      ok_.assign(n_, 1);
      pending_ = n_ - 1;
      ++gen_;
    }
    cv_job_.notify_all();
    ok_[0] = read_share(fd, dst, ranges, 0, share_end(0), &errs_[0]);
    std::unique_lock<std::mutex> lk(m_);
    cv_done_.wait(lk, [this] { return pending_ == 0; });
    for (int i = 0; i < n_; ++i)
      if (!ok_[i]) {
        *err = errs_[i];
        return false;
      }
    return true;
  }

 private:
  uint64_t share_end(int i) const {
    const uint64_t per = ((total_ + parts_ - 1) / parts_ + 4095) & ~4095ull;
    return std::min<uint64_t>(total_, per * (i + 1));
  }

  // Read bytes [b, e) of the concatenated ranges.
  static bool read_share(int fd, uint8_t* dst, const std::vector<Range>& ranges, uint64_t b, uint64_t e,
                         std::string* err) {
    uint64_t pos = 0;
    for (const auto& r : ranges) {
      const uint64_t lo = std::max(b, pos), hi = std::min(e, pos + r.len);
      if (lo < hi && !read_exact(fd, dst + r.at + (lo - pos), hi - lo, r.off + (lo - pos), err)) return false;
      pos += r.len;
      if (pos >= e) break;
    }
    return true;
  }

  void loop(int id) {
    uint64_t seen = 0;
    while (true) {
      std::unique_lock<std::mutex> lk(m_);
      cv_job_.wait(lk, [&] { return stop_ || gen_ != seen; });
      if (stop_) return;
      seen = gen_;
      const bool mine = id < parts_;
      const uint64_t b = mine ? share_end(id - 1) : 0, e = mine ? share_end(id) : 0;
      lk.unlock();
      bool ok = true;
      std::string err;
      if (mine && b < e) ok = read_share(fd_, dst_, *ranges_, b, e, &err);
      lk.lock();
      if (!ok) {
        ok_[id] = 0;
        errs_[id] = err;
      }
      if (--pending_ == 0) cv_done_.notify_one();
    }
  }

  int n_ = 1;
  std::vector<std::thread> workers_;
  std::mutex m_;
  std::condition_variable cv_job_, cv_done_;
  bool stop_ = false;
  uint64_t gen_ = 0;
  int pending_ = 0;
  int fd_ = -1;
  uint8_t* dst_ = nullptr;
  const std::vector<Range>* ranges_ = nullptr;
  uint64_t total_ = 0;
  int parts_ = 1;
  std::vector<std::string> errs_;
  std::vector<char> ok_;
};

}  // namespace stf
}  // namespace tp

struct tp_st_file {
  int fd = -1;
  std::string path;
  uint64_t file_size = 0;
  uint64_t data_start = 0;
  std::vector<tp::stf::Entry> entries;  // in order of increasing offset
  std::unordered_map<std::string, int64_t> index;
  size_t staging_bytes = 0;
  tp_st_read_mode mode = TP_ST_READ_AUTO;
  // Slots: one event each, recorded after the slot's copies; a slot is reused once it fired.
  cudaEvent_t done[2] = {nullptr, nullptr};
  bool pending[2] = {false, false};
  int device = -1;  // the device the events and staging buffers belong to
  int slot = 0;
  // Staged reads: page-locked staging buffers and the reader threads.
  void* staging[2] = {nullptr, nullptr};
  int io_threads = 1;
  std::unique_ptr<tp::stf::ReadPool> pool;
  // Mapped reads: the whole file mapped read-only (map_state 1), or found unusable (-1, reason
  // in map_error); device staging buffers for rowwise loads.
  const uint8_t* map = nullptr;
  int map_state = 0;
  std::string map_error;
  uint64_t page = 4096;
  void* dstage[2] = {nullptr, nullptr};
};

namespace {

using tp::fail;

// The whole pages of the mapping that cover file bytes [off, off + len).
void page_span(const tp_st_file* f, uint64_t off, uint64_t len, uint8_t** start, size_t* bytes) {
  const uint64_t b = off & ~(f->page - 1);
  const uint64_t e = (off + len + f->page - 1) & ~(f->page - 1);
  *start = const_cast<uint8_t*>(f->map) + b;
  *bytes = static_cast<size_t>(e - b);
}

tp_status wait_slot(tp_st_file* f, int s) {
  if (!f->pending[s]) return TP_OK;
  f->pending[s] = false;
  cudaError_t e = cudaEventSynchronize(f->done[s]);
  if (e != cudaSuccess) return tp::cuda_fail(e, "waiting for a shard copy");
  return TP_OK;
}

// Wait for both slots and free the events and staging buffers (the mapping stays).
tp_status release_staging(tp_st_file* f) {
  tp_status st = TP_OK;
  int cur = -1;
  const bool switch_back = f->device >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != f->device &&
                           cudaSetDevice(f->device) == cudaSuccess;
  for (int s = 0; s < 2; ++s) {
    tp_status w = wait_slot(f, s);
    if (st == TP_OK) st = w;
    if (f->done[s]) cudaEventDestroy(f->done[s]);
    if (f->staging[s]) cudaFreeHost(f->staging[s]);
    if (f->dstage[s]) cudaFree(f->dstage[s]);
    f->done[s] = nullptr;
    f->staging[s] = nullptr;
    f->dstage[s] = nullptr;
  }
  if (switch_back) cudaSetDevice(cur);
  f->device = -1;
  return st;
}

// Events on the current device (everything re-made if the device changed), and the buffers a
// load needs: page-locked staging for staged reads, device staging for mapped rowwise reads.
tp_status ensure_slots(tp_st_file* f, bool mapped, bool device_staging) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tp::cuda_fail(e, "cudaGetDevice");
  if (f->device >= 0 && f->device != dev) {
    tp_status st = release_staging(f);
    if (st != TP_OK) return st;
  }
  if (f->done[0] == nullptr) {
    for (int s = 0; s < 2; ++s) {
      e = cudaEventCreateWithFlags(&f->done[s], cudaEventDisableTiming);
      if (e != cudaSuccess) {
        f->done[s] = nullptr;
        release_staging(f);
        return tp::cuda_fail(e, "cudaEventCreate");
      }
    }
    f->device = dev;
  }
  for (int s = 0; s < 2; ++s) {
    if (!mapped && f->staging[s] == nullptr) {
      e = cudaHostAlloc(&f->staging[s], f->staging_bytes, cudaHostAllocPortable);
      if (e != cudaSuccess) {
        f->staging[s] = nullptr;
        release_staging(f);
        return tp::cuda_fail(e, "cudaHostAlloc(staging)");
      }
    }
    if (mapped && device_staging && f->dstage[s] == nullptr) {
      e = cudaMalloc(&f->dstage[s], f->staging_bytes);
      if (e != cudaSuccess) {
        f->dstage[s] = nullptr;
        release_staging(f);
        return tp::cuda_fail(e, "cudaMalloc(device staging)");
      }
    }
  }
  return TP_OK;
}

// Map the file once.  Mapped reads are unusable (map_state -1, reason kept) if the mapping
// fails or the kernel cannot populate a mapping on request.
void ensure_map(tp_st_file* f) {
  if (f->map_state != 0) return;
  const long pg = sysconf(_SC_PAGESIZE);
  f->page = pg > 0 ? static_cast<uint64_t>(pg) : 4096;
  void* m = mmap(nullptr, static_cast<size_t>(f->file_size), PROT_READ, MAP_SHARED, f->fd, 0);
  if (m == MAP_FAILED) {
    f->map_state = -1;
    f->map_error = std::string("mmap failed: ") + strerror(errno);
    return;
  }
  int rc;
  do {
    rc = madvise(m, static_cast<size_t>(std::min<uint64_t>(f->page, f->file_size)), MADV_POPULATE_READ);
  } while (rc != 0 && errno == EINTR);
  if (rc != 0) {
    f->map_error = std::string("madvise(MADV_POPULATE_READ) failed: ") + strerror(errno);
    munmap(m, static_cast<size_t>(f->file_size));
    f->map_state = -1;
    return;
  }
  madvise(m, static_cast<size_t>(std::min<uint64_t>(f->page, f->file_size)), MADV_DONTNEED);
  f->map = static_cast<const uint8_t*>(m);
  f->map_state = 1;
}

// The mode a load on the current device uses (TP_ST_READ_AUTO resolved).
tp_status resolve_mode(tp_st_file* f, tp_st_read_mode* out) {
  *out = TP_ST_READ_STAGED;
  if (f->mode == TP_ST_READ_STAGED) return TP_OK;
  int dev = -1, host_tables = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tp::cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&host_tables, cudaDevAttrPageableMemoryAccessUsesHostPageTables, dev);
  if (e != cudaSuccess) return tp::cuda_fail(e, "cudaDeviceGetAttribute(PageableMemoryAccessUsesHostPageTables)");
  std::string why;
  if (host_tables != 1) {
    why = "device " + std::to_string(dev) + " does not read pageable memory through the host's page tables";
  } else {
    ensure_map(f);
    if (f->map_state != 1) why = f->map_error;
  }
  if (why.empty()) {
    *out = TP_ST_READ_MAPPED;
    return TP_OK;
  }
  if (f->mode == TP_ST_READ_MAPPED)
    return tp::fail(TP_ERR_UNSUPPORTED, "%s: mapped reads are not available: %s", f->path.c_str(), why.c_str());
  return TP_OK;
}

// Fault in the pages of file bytes [off, off + len) (reading them from disk if need be), so
// that the copy engine finds them mapped and a read error surfaces here.  Returns 0 or errno.
int populate(const tp_st_file* f, uint64_t off, uint64_t len) {
  uint8_t* p = nullptr;
  size_t n = 0;
  page_span(f, off, len, &p, &n);
  int rc;
  do {
    rc = madvise(p, n, MADV_POPULATE_READ);
  } while (rc != 0 && errno == EINTR);
  return rc == 0 ? 0 : errno;
}

// Populates the file ranges of a mapped load one ahead of their copies, on a helper thread:
// take(i) waits for range i's pages (and starts range i + 1's).
class PopulateAhead {
 public:
  PopulateAhead(const tp_st_file* f, const char* name, std::vector<std::pair<uint64_t, uint64_t>> ranges)
      : f_(f), name_(name), ranges_(std::move(ranges)) {
    if (!ranges_.empty()) next_ = start(0);
  }
  tp_status take(size_t i) {
    const int err = next_.get();
    if (i + 1 < ranges_.size()) next_ = start(i + 1);
    if (err == 0) return TP_OK;
    return tp::fail(TP_ERR_IO, "%s: tensor \"%s\": cannot read file bytes [%llu, %llu): %s", f_->path.c_str(), name_,
                    (unsigned long long)ranges_[i].first, (unsigned long long)(ranges_[i].first + ranges_[i].second),
                    strerror(err));
  }

 private:
  std::future<int> start(size_t i) {
    const tp_st_file* f = f_;
    const auto r = ranges_[i];
    auto job = [f, r] { return populate(f, r.first, r.second); };
    try {
      return std::async(std::launch::async, job);
    } catch (const std::system_error&) {  // no thread to be had: populate when the range is taken
      return std::async(std::launch::deferred, job);
    }
  }
  const tp_st_file* f_;
  const char* name_;
  std::vector<std::pair<uint64_t, uint64_t>> ranges_;
  std::future<int> next_;
};

// Take the next staging buffer once its previous copy has finished.
tp_status next_slot(tp_st_file* f, int* s) {
  *s = f->slot;
  f->slot ^= 1;
  return wait_slot(f, *s);
}

tp_status mark_slot(tp_st_file* f, int s, cudaStream_t stream) {
  cudaError_t e = cudaEventRecord(f->done[s], stream);
  if (e != cudaSuccess) return tp::cuda_fail(e, "cudaEventRecord");
  f->pending[s] = true;
  return TP_OK;
}

}  // namespace

extern "C" {

size_t tp_st_dtype_size(tp_st_dtype dtype) { return tp::stf::dtype_size(dtype); }

tp_status tp_st_open(const char* path, size_t staging_bytes, tp_st_file** out) {
  using namespace tp;
  clear_error();
  if (out == nullptr) return fail(TP_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (path == nullptr) return fail(TP_ERR_INVALID_ARG, "path is NULL");
  const int fd = open(path, O_RDONLY | O_CLOEXEC);
  if (fd < 0) return fail(TP_ERR_IO, "cannot open %s: %s", path, strerror(errno));
  auto* f = new tp_st_file();
  f->fd = fd;
  f->path = path;
  auto bail = [&](tp_status st) {
    close(f->fd);
    delete f;
    return st;
  };
  struct stat sb {};
  if (fstat(fd, &sb) != 0) return bail(fail(TP_ERR_IO, "cannot stat %s: %s", path, strerror(errno)));
  f->file_size = static_cast<uint64_t>(sb.st_size);
  std::string err;
  uint8_t len8[8];
  if (f->file_size < 8) return bail(fail(TP_ERR_FORMAT, "%s: %llu bytes, shorter than the 8-byte header length", path,
                                         (unsigned long long)f->file_size));
  if (!stf::read_exact(fd, len8, 8, 0, &err)) return bail(fail(TP_ERR_IO, "%s: %s", path, err.c_str()));
  uint64_t n = 0;
  for (int i = 7; i >= 0; --i) n = (n << 8) | len8[i];  // little-endian
  if (n > stf::kMaxHeaderBytes)
    return bail(fail(TP_ERR_FORMAT, "%s: header of %llu bytes exceeds the %llu-byte limit", path,
                     (unsigned long long)n, (unsigned long long)stf::kMaxHeaderBytes));
  if (8 + n > f->file_size)
    return bail(fail(TP_ERR_FORMAT, "%s: header of %llu bytes runs past the end of the %llu-byte file", path,
                     (unsigned long long)n, (unsigned long long)f->file_size));
  std::string header(static_cast<size_t>(n), '\0');
  if (n > 0 && !stf::read_exact(fd, &header[0], n, 8, &err)) return bail(fail(TP_ERR_IO, "%s: %s", path, err.c_str()));
  f->data_start = 8 + n;
  const uint64_t data_size = f->file_size - f->data_start;

  stf::Json js(header);
  if (!js.expect('{')) return bail(fail(TP_ERR_FORMAT, "%s: %s", path, js.error().c_str()));
  bool meta_seen = false;
  if (!js.peek('}')) {
    while (true) {
      std::string key;
      if (!js.string(&key) || !js.expect(':')) return bail(fail(TP_ERR_FORMAT, "%s: %s", path, js.error().c_str()));
      if (key == "__metadata__") {
        if (meta_seen) return bail(fail(TP_ERR_FORMAT, "%s: two __metadata__ entries", path));
        meta_seen = true;
        if (!js.skip_value(1)) return bail(fail(TP_ERR_FORMAT, "%s: %s", path, js.error().c_str()));
      } else {
        stf::Entry t;
        t.name = key;
        if (!js.tensor(&t))
          return bail(fail(TP_ERR_FORMAT, "%s: tensor \"%s\": %s", path, key.c_str(), js.error().c_str()));
        if (f->index.count(key)) return bail(fail(TP_ERR_FORMAT, "%s: tensor \"%s\" appears twice", path, key.c_str()));
        if (t.begin > t.end || t.end > data_size)
          return bail(fail(TP_ERR_FORMAT, "%s: tensor \"%s\": data_offsets [%llu, %llu] outside the %llu data bytes",
                           path, key.c_str(), (unsigned long long)t.begin, (unsigned long long)t.end,
                           (unsigned long long)data_size));
        uint64_t bytes = stf::dtype_size(t.dtype);
        for (int d = 0; d < t.ndim; ++d) {
          const uint64_t dim = static_cast<uint64_t>(t.shape[d]);
          if (dim != 0 && bytes > UINT64_MAX / dim)
            return bail(fail(TP_ERR_FORMAT, "%s: tensor \"%s\": shape overflows", path, key.c_str()));
          bytes *= dim;
        }
        if (bytes != t.end - t.begin)
          return bail(fail(TP_ERR_FORMAT, "%s: tensor \"%s\": shape needs %llu bytes, data_offsets give %llu", path,
                           key.c_str(), (unsigned long long)bytes, (unsigned long long)(t.end - t.begin)));
        f->index[key] = 0;
        f->entries.push_back(std::move(t));
      }
      if (js.peek(',')) {
        js.expect(',');
        continue;
      }
      break;
    }
  }
  if (!js.expect('}')) return bail(fail(TP_ERR_FORMAT, "%s: %s", path, js.error().c_str()));
  if (!js.at_end()) return bail(fail(TP_ERR_FORMAT, "%s: text after the header object", path));

  std::stable_sort(f->entries.begin(), f->entries.end(),
                   [](const stf::Entry& a, const stf::Entry& b) { return a.begin < b.begin; });
  uint64_t prev_end = 0;
  const stf::Entry* prev = nullptr;
  for (size_t i = 0; i < f->entries.size(); ++i) {
    const stf::Entry& t = f->entries[i];
    if (t.end > t.begin) {
      if (prev != nullptr && t.begin < prev_end)
        return bail(fail(TP_ERR_FORMAT, "%s: tensors \"%s\" and \"%s\" overlap", path, prev->name.c_str(),
                         t.name.c_str()));
      prev_end = t.end;
      prev = &t;
    }
    f->index[t.name] = static_cast<int64_t>(i);
  }
  size_t sb_bytes = staging_bytes == 0 ? TP_ST_DEFAULT_STAGING_BYTES : staging_bytes;
  sb_bytes = (std::max<size_t>(sb_bytes, 4096) + 4095) & ~static_cast<size_t>(4095);
  f->staging_bytes = sb_bytes;
  const unsigned hw = std::thread::hardware_concurrency();
  f->io_threads = static_cast<int>(std::min(16u, std::max(1u, hw)));
  *out = f;
  return TP_OK;
}

tp_status tp_st_close(tp_st_file* file) {
  tp::clear_error();
  if (file == nullptr) return TP_OK;
  tp_status st = release_staging(file);
  if (file->map != nullptr) munmap(const_cast<uint8_t*>(file->map), static_cast<size_t>(file->file_size));
  if (file->fd >= 0) close(file->fd);
  delete file;
  return st;
}

tp_status tp_st_set_read_mode(tp_st_file* file, tp_st_read_mode mode) {
  tp::clear_error();
  if (file == nullptr) return tp::fail(TP_ERR_INVALID_ARG, "file is NULL");
  if (mode != TP_ST_READ_AUTO && mode != TP_ST_READ_STAGED && mode != TP_ST_READ_MAPPED)
    return tp::fail(TP_ERR_INVALID_ARG, "read mode %d is not a tp_st_read_mode", static_cast<int>(mode));
  file->mode = mode;
  return TP_OK;
}

tp_status tp_st_read_mode_on_device(tp_st_file* file, tp_st_read_mode* mode) {
  tp::clear_error();
  if (file == nullptr || mode == nullptr) return tp::fail(TP_ERR_INVALID_ARG, "file or mode is NULL");
  return resolve_mode(file, mode);
}

int64_t tp_st_count(const tp_st_file* file) {
  return file == nullptr ? -1 : static_cast<int64_t>(file->entries.size());
}

tp_status tp_st_info(const tp_st_file* file, int64_t index, const char** name, tp_st_dtype* dtype, int* ndim,
                     int64_t* shape, uint64_t* offset, uint64_t* nbytes) {
  using namespace tp;
  clear_error();
  if (file == nullptr) return fail(TP_ERR_INVALID_ARG, "file is NULL");
  if (index < 0 || index >= static_cast<int64_t>(file->entries.size()))
    return fail(TP_ERR_INVALID_ARG, "tensor index %lld outside [0, %zu)", (long long)index, file->entries.size());
  const stf::Entry& t = file->entries[static_cast<size_t>(index)];
  if (name) *name = t.name.c_str();
  if (dtype) *dtype = t.dtype;
  if (ndim) *ndim = t.ndim;
  if (shape)
    for (int d = 0; d < t.ndim; ++d) shape[d] = t.shape[d];
  if (offset) *offset = file->data_start + t.begin;
  if (nbytes) *nbytes = t.end - t.begin;
  return TP_OK;
}

int64_t tp_st_find(const tp_st_file* file, const char* name) {
  if (file == nullptr || name == nullptr) return -1;
  auto it = file->index.find(name);
  return it == file->index.end() ? -1 : it->second;
}

tp_status tp_st_plan_shard_ranks(tp_st_file* file, const char* name, tp_style style, int tp_degree, int rank_begin,
                                 int rank_count, const int64_t* fused_splits, int n_splits, int64_t num_heads,
                                 int64_t head_dim, void* const* dev_outs, tp_stream_t stream) {
  using namespace tp;
  clear_error();
  if (file == nullptr || name == nullptr) return fail(TP_ERR_INVALID_ARG, "file or name is NULL");
  const int64_t idx = tp_st_find(file, name);
  if (idx < 0) return fail(TP_ERR_NOT_FOUND, "no tensor \"%s\" in %s", name, file->path.c_str());
  const stf::Entry& t = file->entries[static_cast<size_t>(idx)];
  const int64_t esz = static_cast<int64_t>(stf::dtype_size(t.dtype));

  // The tensor as a matrix [rows, cols] of elements.
  int64_t rows = 1, cols = 1;
  if (t.ndim == 1) {
    if (style == TP_ROWWISE)
      return fail(TP_ERR_INVALID_ARG, "tensor \"%s\" is 1-D: it has no dim 1 to shard rowwise (load it with "
                  "tp_degree 1 to replicate it)", name);
    rows = t.shape[0];
  } else if (t.ndim >= 2) {
    if (style == TP_ROWWISE && t.ndim > 2)
      return fail(TP_ERR_UNSUPPORTED, "rowwise sharding of the %d-D tensor \"%s\"", t.ndim, name);
    rows = t.shape[0];
    for (int d = 1; d < t.ndim; ++d) cols *= t.shape[d];
  }
  if (rank_count < 0) return fail(TP_ERR_INVALID_ARG, "rank_count %d is negative", rank_count);
  if (rank_begin < 0) return fail(TP_ERR_INVALID_ARG, "rank %d is negative", rank_begin);
  int64_t sizes[TP_MAX_SPLITS];
  int n = 0;
  tp_status st = validate_plan(rows, cols, style, tp_degree, rank_count > 0 ? rank_begin : -1, num_heads, head_dim,
                               fused_splits, n_splits, sizes, &n);
  if (st != TP_OK) return st;
  // rank_begin is in [0, tp_degree) here (validate_plan checked it), so the difference cannot overflow.
  if (rank_count > 0 && rank_count > tp_degree - rank_begin)
    return fail(TP_ERR_INVALID_ARG, "ranks [%d, %lld) outside [0, %d)", rank_begin,
                static_cast<long long>(rank_begin) + rank_count, tp_degree);
  const int64_t row_bytes = cols * esz;
  if (style == TP_ROWWISE) {
    // The extraction kernel moves 16-bit units: every column segment must be whole units.
    bool even = (row_bytes % 2) == 0;
    for (int b = 0; b < n; ++b) even = even && ((sizes[b] / tp_degree) * esz) % 2 == 0;
    if (!even)
      return fail(TP_ERR_UNSUPPORTED, "rowwise slices of \"%s\" are an odd number of bytes wide", name);
    if (static_cast<uint64_t>(row_bytes) > file->staging_bytes)
      return fail(TP_ERR_UNSUPPORTED, "a row of \"%s\" (%lld bytes) does not fit the %zu-byte staging buffer; open "
                  "the file with a larger staging size", name, (long long)row_bytes, file->staging_bytes);
  }
  if (rank_count == 0 || rows == 0 || cols == 0) return TP_OK;
  if (dev_outs == nullptr) return fail(TP_ERR_INVALID_ARG, "dev_outs is NULL");
  for (int i = 0; i < rank_count; ++i) {
    if (dev_outs[i] == nullptr) return fail(TP_ERR_INVALID_ARG, "dev_outs[%d] is NULL", i);
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, dev_outs[i]);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(dev_out)");
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
      return fail(TP_ERR_INVALID_ARG, "dev_outs[%d] is not device memory", i);
  }
  tp_st_read_mode mode = TP_ST_READ_STAGED;
  st = resolve_mode(file, &mode);
  if (st != TP_OK) return st;
  const bool mapped = mode == TP_ST_READ_MAPPED;
  st = ensure_slots(file, mapped, style == TP_ROWWISE);
  if (st != TP_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint64_t base = file->data_start + t.begin;
  const uint64_t chunk = file->staging_bytes;
  std::string err;

  if (!mapped && !file->pool) file->pool.reset(new stf::ReadPool(file->io_threads));

  if (style == TP_COLWISE) {
    // Rank r's part of block b: rows [o_b + r*s_b/p, o_b + (r+1)*s_b/p), one byte range of the
    // file, landing at rows [sum_{b'<b} s_b'/p, ...) of the rank's shard.  The pieces are packed
    // back to back into the staging buffers (a piece may straddle two), each buffer read in one
    // parallel job and copied out with one cudaMemcpyAsync per piece.
    struct Piece {
      uint64_t src, len;
      uint8_t* dst;
    };
    std::vector<Piece> pieces;
    for (int i = 0; i < rank_count; ++i) {
      const int rank = rank_begin + i;
      uint8_t* dst = static_cast<uint8_t*>(dev_outs[i]);
      int64_t block_off = 0, out_row = 0;
      for (int b = 0; b < n; ++b) {
        const int64_t part = sizes[b] / tp_degree;
        Piece pc{base + static_cast<uint64_t>((block_off + rank * part) * row_bytes),
                 static_cast<uint64_t>(part * row_bytes), dst + out_row * row_bytes};
        if (!pieces.empty() && pieces.back().src + pieces.back().len == pc.src &&
            pieces.back().dst + pieces.back().len == pc.dst)
          pieces.back().len += pc.len;  // contiguous in the file and in the shard
        else if (pc.len > 0)
          pieces.push_back(pc);
        block_off += sizes[b];
        out_row += part;
      }
    }
    if (mapped) {
      // Each piece is populated, then copied by the copy engine straight from the mapping; a
      // slot's event marks the end, so that closing the file waits for the copies.
      int slot = 0;
      st = next_slot(file, &slot);
      if (st != TP_OK) return st;
      std::vector<std::pair<uint64_t, uint64_t>> spans;
      for (const Piece& pc : pieces) spans.emplace_back(pc.src, pc.len);
      PopulateAhead ahead(file, name, std::move(spans));
      for (size_t i = 0; i < pieces.size(); ++i) {
        const Piece& pc = pieces[i];
        st = ahead.take(i);
        if (st != TP_OK) return st;
        cudaError_t e = cudaMemcpyAsync(pc.dst, file->map + pc.src, pc.len, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(mapped file to shard)");
      }
      return mark_slot(file, slot, s);
    }
    std::vector<stf::Range> ranges;
    std::vector<std::pair<uint8_t*, stf::Range>> copies;
    uint64_t used = 0;
    auto flush = [&]() -> tp_status {
      if (ranges.empty()) return TP_OK;
      int slot = 0;
      tp_status rc = next_slot(file, &slot);
      if (rc != TP_OK) return rc;
      uint8_t* stage = static_cast<uint8_t*>(file->staging[slot]);
      if (!file->pool->run(file->fd, stage, ranges, &err))
        return fail(TP_ERR_IO, "%s: tensor \"%s\": %s", file->path.c_str(), name, err.c_str());
      for (const auto& c : copies) {
        cudaError_t e = cudaMemcpyAsync(c.first, stage + c.second.at, c.second.len, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(staging to shard)");
      }
      rc = mark_slot(file, slot, s);
      ranges.clear();
      copies.clear();
      used = 0;
      return rc;
    };
    for (const Piece& pc : pieces) {
      uint64_t src = pc.src, left = pc.len;
      uint8_t* d = pc.dst;
      while (left > 0) {
        const uint64_t len = std::min(left, chunk - used);
        const stf::Range r{src, len, used};
        ranges.push_back(r);
        copies.emplace_back(d, r);
        used += len;
        src += len;
        d += len;
        left -= len;
        if (used == chunk) {
          st = flush();
          if (st != TP_OK) return st;
        }
      }
    }
    return flush();
  }

  // Rowwise: whole rows in chunks; the ranks' column segments are extracted on the GPU.
  const int64_t units = row_bytes / 2;
  int64_t unit_sizes[TP_MAX_SPLITS];
  for (int b = 0; b < n; ++b) unit_sizes[b] = sizes[b] * esz / 2;
  const int64_t shard_row_bytes = row_bytes / tp_degree;
  const int64_t chunk_rows = static_cast<int64_t>(chunk / static_cast<uint64_t>(row_bytes));
  void* outs[TP_MAX_DEGREE > 64 ? TP_MAX_DEGREE : 64];
  if (rank_count > static_cast<int>(sizeof(outs) / sizeof(outs[0])))
    return fail(TP_ERR_UNSUPPORTED, "%d ranks in one rowwise load", rank_count);
  std::unique_ptr<PopulateAhead> ahead;
  if (mapped) {
    std::vector<std::pair<uint64_t, uint64_t>> spans;
    for (int64_t r0 = 0; r0 < rows; r0 += chunk_rows)
      spans.emplace_back(base + static_cast<uint64_t>(r0 * row_bytes),
                         static_cast<uint64_t>(std::min(chunk_rows, rows - r0) * row_bytes));
    ahead.reset(new PopulateAhead(file, name, std::move(spans)));
  }
  for (int64_t r0 = 0; r0 < rows; r0 += chunk_rows) {
    const int64_t nr = std::min(chunk_rows, rows - r0);
    int slot = 0;
    st = next_slot(file, &slot);
    if (st != TP_OK) return st;
    const uint64_t off = base + static_cast<uint64_t>(r0 * row_bytes), len = static_cast<uint64_t>(nr * row_bytes);
    void* rows_buf = nullptr;
    if (mapped) {
      // The rows go to a device staging buffer; the extraction kernel then reads device memory.
      st = ahead->take(static_cast<size_t>(r0 / chunk_rows));
      if (st != TP_OK) return st;
      cudaError_t e = cudaMemcpyAsync(file->dstage[slot], file->map + off, len, cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(mapped file to device staging)");
      rows_buf = file->dstage[slot];
    } else {
      const std::vector<stf::Range> rows_range{{off, len, 0}};
      if (!file->pool->run(file->fd, static_cast<uint8_t*>(file->staging[slot]), rows_range, &err))
        return fail(TP_ERR_IO, "%s: tensor \"%s\": %s", file->path.c_str(), name, err.c_str());
      rows_buf = file->staging[slot];
    }
    for (int i = 0; i < rank_count; ++i) outs[i] = static_cast<uint8_t*>(dev_outs[i]) + r0 * shard_row_bytes;
    st = tp_plan_shard_ranks(rows_buf, nr, units, TP_ROWWISE, tp_degree, rank_begin, rank_count,
                             n_splits > 0 ? unit_sizes : nullptr, n_splits > 0 ? n : 0, 0, 0, outs, stream);
    if (st != TP_OK) return st;
    st = mark_slot(file, slot, s);
    if (st != TP_OK) return st;
  }
  return TP_OK;
}

}  // extern "C"
