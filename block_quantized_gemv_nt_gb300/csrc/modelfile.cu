// Model files: the host-file tier of the three-tier cache ("Ntransformer"
// (en.unwiki.net), About: VRAM-resident layers, pinned RAM, NVMe / mmap
// fallback) and its "mmap pinned" data path ("ntransformer - moteur
// d'inférence NVMe-to-GPU…" (fr.news.hada.io), "Fonctionnalités
// principales": resident > H2D from pinned RAM > mmap pinned > CPU memcpy).
//
// The native reader of the container the Python writer produces:
//
//   offset 0   "NTQF", u32 version (1), u64 header length H (little-endian)
//   offset 16  H bytes of JSON: {"spec": {...}, "blob_offsets": [7 ints],
//              "blob_bytes": int, "entries": {name: [offset, bytes], ...}}
//   data       entries at 4096-byte-aligned offsets from the first 4096
//              boundary after the header: "embd", "out", "out_norm", and
//              per layer l "blob.l" (its seven matrices in the blob layout
//              of nt_layer_blob_layout), "attn_norm.l", "ffn_norm.l".
//
// Host code only: the file is mapped read-only and checked before any entry
// is handed out; page-locking goes through cudaHostRegister / cudaHostAlloc.
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <atomic>
#include <charconv>
#include <cstring>
#include <map>
#include <string>
#include <utility>
#include <vector>

#include "nt_internal.cuh"

namespace nt {
extern thread_local std::string g_create_error;
}

namespace {

constexpr uint64_t kFileAlign = 4096;  // entry alignment in the file, and the page-lock granule
constexpr int kMaxJsonDepth = 32;

// test hook (nt_debug_file_refuse_in_place): treat both in-place rungs as
// refused, so nt_file_lock takes the CPU copy (process-wide)
std::atomic<int> g_refuse_in_place{0};

uint64_t up(uint64_t n, uint64_t a) { return (n + a - 1) / a * a; }

// ---- a JSON reader (RFC 8259) for the header --------------------------------

struct JVal {
  enum Kind { kNull, kBool, kNum, kStr, kArr, kObj } kind = kNull;
  bool b = false;
  double num = 0;
  bool is_int = false;  // an integer literal that fits int64
  int64_t i = 0;
  std::string s;
  std::vector<JVal> a;
  std::vector<std::pair<std::string, JVal>> o;

  const JVal* get(const char* key) const {
    if (kind != kObj) return nullptr;
    for (const auto& kv : o)
      if (kv.first == key) return &kv.second;
    return nullptr;
  }
};

class JsonReader {
 public:
  JsonReader(const char* p, size_t n) : p_(p), e_(p + n) {}

  // the whole text is one value, with only white space around it
  bool document(JVal& v) {
    ws();
    if (!value(v, 0)) return false;
    ws();
    return p_ == e_;
  }

 private:
  const char* p_;
  const char* e_;

  void ws() {
    while (p_ < e_ && (*p_ == ' ' || *p_ == '\t' || *p_ == '\n' || *p_ == '\r')) ++p_;
  }
  bool word(const char* w) {
    const size_t n = strlen(w);
    if (size_t(e_ - p_) < n || memcmp(p_, w, n) != 0) return false;
    p_ += n;
    return true;
  }
  bool value(JVal& v, int depth) {
    if (p_ >= e_ || depth > kMaxJsonDepth) return false;
    switch (*p_) {
      case '{': return object(v, depth);
      case '[': return array(v, depth);
      case '"': v.kind = JVal::kStr; return string(v.s);
      case 't': v.kind = JVal::kBool; v.b = true; return word("true");
      case 'f': v.kind = JVal::kBool; v.b = false; return word("false");
      case 'n': v.kind = JVal::kNull; return word("null");
      default: return number(v);
    }
  }
  bool object(JVal& v, int depth) {
    v.kind = JVal::kObj;
    ++p_;
    ws();
    if (p_ < e_ && *p_ == '}') return ++p_, true;
    for (;;) {
      std::string key;
      JVal x;
      ws();
      if (p_ >= e_ || *p_ != '"' || !string(key)) return false;
      ws();
      if (p_ >= e_ || *p_++ != ':') return false;
      ws();
      if (!value(x, depth + 1)) return false;
      v.o.emplace_back(std::move(key), std::move(x));
      ws();
      if (p_ >= e_) return false;
      const char c = *p_++;
      if (c == '}') return true;
      if (c != ',') return false;
    }
  }
  bool array(JVal& v, int depth) {
    v.kind = JVal::kArr;
    ++p_;
    ws();
    if (p_ < e_ && *p_ == ']') return ++p_, true;
    for (;;) {
      JVal x;
      ws();
      if (!value(x, depth + 1)) return false;
      v.a.push_back(std::move(x));
      ws();
      if (p_ >= e_) return false;
      const char c = *p_++;
      if (c == ']') return true;
      if (c != ',') return false;
    }
  }
  bool hex4(unsigned& u) {
    if (e_ - p_ < 4) return false;
    u = 0;
    for (int k = 0; k < 4; ++k) {
      const char c = *p_++;
      const int d = c >= '0' && c <= '9' ? c - '0' : c >= 'a' && c <= 'f' ? c - 'a' + 10
                  : c >= 'A' && c <= 'F' ? c - 'A' + 10 : -1;
      if (d < 0) return false;
      u = u * 16 + unsigned(d);
    }
    return true;
  }
  static void utf8(std::string& s, unsigned u) {
    if (u < 0x80) {
      s.push_back(char(u));
    } else if (u < 0x800) {
      s.push_back(char(0xC0 | (u >> 6)));
      s.push_back(char(0x80 | (u & 0x3F)));
    } else if (u < 0x10000) {
      s.push_back(char(0xE0 | (u >> 12)));
      s.push_back(char(0x80 | ((u >> 6) & 0x3F)));
      s.push_back(char(0x80 | (u & 0x3F)));
    } else {
      s.push_back(char(0xF0 | (u >> 18)));
      s.push_back(char(0x80 | ((u >> 12) & 0x3F)));
      s.push_back(char(0x80 | ((u >> 6) & 0x3F)));
      s.push_back(char(0x80 | (u & 0x3F)));
    }
  }
  bool string(std::string& s) {
    ++p_;  // the opening quote
    while (p_ < e_) {
      const unsigned char c = static_cast<unsigned char>(*p_++);
      if (c == '"') return true;
      if (c < 0x20) return false;  // control characters must be escaped
      if (c != '\\') {
        s.push_back(char(c));
        continue;
      }
      if (p_ >= e_) return false;
      switch (*p_++) {
        case '"': s.push_back('"'); break;
        case '\\': s.push_back('\\'); break;
        case '/': s.push_back('/'); break;
        case 'b': s.push_back('\b'); break;
        case 'f': s.push_back('\f'); break;
        case 'n': s.push_back('\n'); break;
        case 'r': s.push_back('\r'); break;
        case 't': s.push_back('\t'); break;
        case 'u': {
          unsigned u = 0, lo = 0;
          if (!hex4(u)) return false;
          if (u >= 0xD800 && u < 0xDC00) {  // a high surrogate takes a low one after it
            if (!word("\\u") || !hex4(lo) || lo < 0xDC00 || lo >= 0xE000) return false;
            u = 0x10000 + ((u - 0xD800) << 10) + (lo - 0xDC00);
          } else if (u >= 0xDC00 && u < 0xE000) {
            return false;
          }
          utf8(s, u);
          break;
        }
        default: return false;
      }
    }
    return false;
  }
  static bool digit(char c) { return c >= '0' && c <= '9'; }
  bool number(JVal& v) {
    const char* b = p_;
    if (p_ < e_ && *p_ == '-') ++p_;
    if (p_ >= e_) return false;
    if (*p_ == '0') {
      ++p_;
    } else if (*p_ >= '1' && *p_ <= '9') {
      while (p_ < e_ && digit(*p_)) ++p_;
    } else {
      return false;
    }
    bool integral = true;
    if (p_ < e_ && *p_ == '.') {
      integral = false;
      ++p_;
      if (p_ >= e_ || !digit(*p_)) return false;
      while (p_ < e_ && digit(*p_)) ++p_;
    }
    if (p_ < e_ && (*p_ == 'e' || *p_ == 'E')) {
      integral = false;
      ++p_;
      if (p_ < e_ && (*p_ == '+' || *p_ == '-')) ++p_;
      if (p_ >= e_ || !digit(*p_)) return false;
      while (p_ < e_ && digit(*p_)) ++p_;
    }
    v.kind = JVal::kNum;
    // from_chars: locale-independent, and exact for the integers
    if (std::from_chars(b, p_, v.num).ec != std::errc()) return false;
    if (integral) v.is_int = std::from_chars(b, p_, v.i).ec == std::errc();
    return true;
  }
};

// ---- the header's fields ------------------------------------------------------

bool get_int(const JVal* o, const char* key, int64_t lo, int64_t hi, int64_t& out) {
  const JVal* v = o ? o->get(key) : nullptr;
  if (!v || v->kind != JVal::kNum || !v->is_int || v->i < lo || v->i > hi) return false;
  out = v->i;
  return true;
}

bool get_num(const JVal* o, const char* key, double& out) {
  const JVal* v = o ? o->get(key) : nullptr;
  if (!v || v->kind != JVal::kNum) return false;
  out = v->num;
  return true;
}

size_t matrix_bytes(int fmt, int64_t rows, int64_t cols) {
  return size_t(rows) * size_t(cols / nt::block_elems(fmt)) * size_t(nt::block_bytes(fmt));
}

struct Entry {
  uint64_t off = 0;  // from the start of the file
  uint64_t bytes = 0;
};

struct Lock {
  int rung = 0;
  void* ptr = nullptr;  // the page-locked copy source handed out
  void* map = nullptr;  // a private mapping (rung 1)
  size_t map_len = 0;
};

}  // namespace

struct nt_file {
  int fd = -1;
  uint8_t* base = nullptr;  // the read-only shared mapping of the whole file
  size_t size = 0;
  std::string header;
  nt_model_desc desc{};
  std::map<std::string, Entry> entries;
  std::map<std::string, Lock> locks;
};

namespace {

void release(nt_file* f) {
  if (f->base) munmap(f->base, f->size);
  if (f->fd >= 0) close(f->fd);
  delete f;
}

// every check of a freshly mapped file; an empty string when it passes
std::string index_file(nt_file* f) {
  if (f->size < 16) return "shorter than its 16-byte preamble";
  if (memcmp(f->base, "NTQF", 4) != 0) return "not a model file (magic)";
  uint32_t version = 0;
  uint64_t hlen = 0;
  memcpy(&version, f->base + 4, 4);  // little-endian on both host architectures
  memcpy(&hlen, f->base + 8, 8);
  if (version != 1) return "version " + std::to_string(version) + " (this reader knows 1)";
  if (hlen > f->size - 16) return "the header runs past the end of the file";
  f->header.assign(reinterpret_cast<const char*>(f->base) + 16, size_t(hlen));
  JVal root;
  if (!JsonReader(f->header.data(), f->header.size()).document(root)) return "the header is not valid JSON";
  if (root.kind != JVal::kObj) return "the header is not a JSON object";
  const JVal* spec = root.get("spec");
  const JVal* fmt = spec ? spec->get("fmt") : nullptr;
  if (!spec || spec->kind != JVal::kObj || !fmt || fmt->kind != JVal::kObj) return "the header has no spec / fmt";

  nt_model_desc& d = f->desc;
  int64_t v[7];
  const char* dims[7] = {"n_layers", "d_model", "n_qh", "n_kvh", "head_dim", "ffn", "vocab"};
  for (int k = 0; k < 7; ++k)
    if (!get_int(spec, dims[k], 1, INT32_MAX, v[k])) return std::string("spec.") + dims[k] + " missing or out of range";
  d.n_layers = int(v[0]), d.d_model = int(v[1]), d.n_qh = int(v[2]), d.n_kvh = int(v[3]);
  d.head_dim = int(v[4]), d.ffn = int(v[5]), d.vocab = int(v[6]);
  if (d.n_qh % d.n_kvh) return "spec.n_qh is not a multiple of spec.n_kvh";
  double eps = 0, theta = 0;
  if (!get_num(spec, "eps", eps) || !get_num(spec, "theta", theta) || !(eps > 0) || !(theta > 0))
    return "spec.eps / spec.theta missing or not positive";
  d.eps = float(eps), d.theta = float(theta);
  d.kv_cap = 0;        // the KV cache is runtime state, not part of the file
  d.stream_slots = 0;  // a runtime choice too
  const char* names[9] = {"wq", "wk", "wv", "wo", "wg", "wu", "wd", "embd", "out"};
  int* slots[9] = {&d.fmt_q, &d.fmt_k, &d.fmt_v, &d.fmt_o, &d.fmt_gate, &d.fmt_up, &d.fmt_down, &d.fmt_embd, &d.fmt_out};
  for (int k = 0; k < 9; ++k) {
    int64_t x = 0;
    if (!get_int(fmt, names[k], 0, NT_F32, x)) return std::string("spec.fmt.") + names[k] + " missing or unknown";
    *slots[k] = int(x);
  }
  // every matrix's rows are whole blocks: columns d_model, except wo (n_qh * head_dim) and wd (ffn)
  const int64_t qdim = int64_t(d.n_qh) * d.head_dim;
  for (int k = 0; k < 9; ++k) {
    const int64_t cols = k == 3 ? qdim : k == 6 ? d.ffn : d.d_model;
    if (cols % nt::block_elems(*slots[k])) return std::string(names[k]) + ": columns not a multiple of the block size";
  }
  size_t offs[7], blob = 0;
  if (nt_layer_blob_layout(&d, offs, &blob) != NT_OK) return "the spec has no blob layout";
  const JVal* bo = root.get("blob_offsets");
  if (!bo || bo->kind != JVal::kArr || bo->a.size() != 7) return "blob_offsets is not a list of 7";
  for (int k = 0; k < 7; ++k)
    if (bo->a[k].kind != JVal::kNum || !bo->a[k].is_int || uint64_t(bo->a[k].i) != offs[k])
      return "blob_offsets differ from this library's blob layout";
  int64_t bb = 0;
  if (!get_int(&root, "blob_bytes", 0, INT64_MAX, bb) || uint64_t(bb) != blob)
    return "blob_bytes differs from this library's blob layout";

  const JVal* ents = root.get("entries");
  if (!ents || ents->kind != JVal::kObj) return "the header has no entries";
  const uint64_t data0 = up(16 + hlen, kFileAlign);
  for (const auto& kv : ents->o) {
    const JVal& e = kv.second;
    if (e.kind != JVal::kArr || e.a.size() != 2 || e.a[0].kind != JVal::kNum || !e.a[0].is_int || e.a[0].i < 0 ||
        e.a[1].kind != JVal::kNum || !e.a[1].is_int || e.a[1].i < 0)
      return "entry " + kv.first + " is not [offset, bytes]";
    const uint64_t off = uint64_t(e.a[0].i), n = uint64_t(e.a[1].i);
    // the entry, rounded up to whole 4096-byte units (what page-locking covers), lies inside the file
    if (off > f->size || data0 > f->size - off || n > f->size || up(n, kFileAlign) > f->size - data0 - off)
      return "entry " + kv.first + " runs past the end of the file";
    if ((data0 + off) % kFileAlign) return "entry " + kv.first + " is not 4096-byte aligned";
    if (!f->entries.emplace(kv.first, Entry{data0 + off, n}).second) return "entry " + kv.first + " is listed twice";
  }
  // the entries a model needs, with the sizes its shapes give
  const auto need = [&](const std::string& name, uint64_t bytes, bool at_least) -> std::string {
    const auto it = f->entries.find(name);
    if (it == f->entries.end()) return "entry " + name + " is missing";
    if (at_least ? it->second.bytes < bytes : it->second.bytes != bytes)
      return "entry " + name + " has " + std::to_string(it->second.bytes) + " bytes, expected " +
             (at_least ? "at least " : "") + std::to_string(bytes);
    return "";
  };
  std::string err;
  const uint64_t norm = 4ull * uint64_t(d.d_model);
  if (!(err = need("embd", matrix_bytes(d.fmt_embd, d.vocab, d.d_model), false)).empty()) return err;
  if (!(err = need("out", matrix_bytes(d.fmt_out, d.vocab, d.d_model), false)).empty()) return err;
  if (!(err = need("out_norm", norm, false)).empty()) return err;
  for (int l = 0; l < d.n_layers; ++l) {
    const std::string s = std::to_string(l);
    if (!(err = need("blob." + s, blob, true)).empty()) return err;
    if (!(err = need("attn_norm." + s, norm, false)).empty()) return err;
    if (!(err = need("ffn_norm." + s, norm, false)).empty()) return err;
  }
  return "";
}

}  // namespace

using nt::set_err;

extern "C" {

nt_status nt_file_open(const char* path, nt_file** out) {
  nt::g_create_error.clear();
  if (!path || !out) {
    nt::g_create_error = "nt_file_open: null pointer";
    return NT_ERR_INVALID_ARG;
  }
  *out = nullptr;
  nt_file* f = new nt_file;
  f->fd = open(path, O_RDONLY | O_CLOEXEC);
  struct stat sb {};
  if (f->fd < 0 || fstat(f->fd, &sb) != 0 || !S_ISREG(sb.st_mode)) {
    nt::g_create_error = std::string(path) + ": " + (f->fd < 0 ? strerror(errno) : "not a regular file");
    release(f);
    return NT_ERR_INVALID_ARG;
  }
  f->size = size_t(sb.st_size);
  if (f->size > 0) {
    void* m = mmap(nullptr, f->size, PROT_READ, MAP_SHARED, f->fd, 0);
    if (m == MAP_FAILED) {
      nt::g_create_error = std::string(path) + ": mmap: " + strerror(errno);
      release(f);
      return NT_ERR_INVALID_ARG;
    }
    f->base = static_cast<uint8_t*>(m);
  }
  const std::string err = index_file(f);
  if (!err.empty()) {
    nt::g_create_error = std::string(path) + ": " + err;
    release(f);
    return NT_ERR_INVALID_ARG;
  }
  *out = f;
  return NT_OK;
}

nt_status nt_file_close(nt_file* f) {
  if (!f) {
    nt::g_create_error = "nt_file_close: null file";
    return NT_ERR_INVALID_ARG;
  }
  if (!f->locks.empty()) {
    nt::g_create_error = "nt_file_close: " + std::to_string(f->locks.size()) + " entries are still page-locked";
    return NT_ERR_INVALID_ARG;
  }
  release(f);
  return NT_OK;
}

nt_status nt_file_desc(const nt_file* f, nt_model_desc* desc) {
  if (!f || !desc) return NT_ERR_INVALID_ARG;
  *desc = f->desc;
  return NT_OK;
}

nt_status nt_file_header(const nt_file* f, const char** text, size_t* len) {
  if (!f || !text) return NT_ERR_INVALID_ARG;
  *text = f->header.c_str();
  if (len) *len = f->header.size();
  return NT_OK;
}

nt_status nt_file_entry(const nt_file* f, const char* name, const void** host_ptr, uint64_t* offset, size_t* bytes) {
  if (!f || !name) return NT_ERR_INVALID_ARG;
  const auto it = f->entries.find(name);
  if (it == f->entries.end()) return NT_ERR_INVALID_ARG;
  if (host_ptr) *host_ptr = f->base + it->second.off;
  if (offset) *offset = it->second.off;
  if (bytes) *bytes = size_t(it->second.bytes);
  return NT_OK;
}

nt_status nt_file_lock(nt_ctx* ctx, nt_file* f, const char* name, int allow_copy, const void** pinned_out,
                       int* rung_out) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  if (!f || !name || !pinned_out) return set_err(ctx, NT_ERR_INVALID_ARG, "null pointer");
  const auto it = f->entries.find(name);
  if (it == f->entries.end()) return set_err(ctx, NT_ERR_INVALID_ARG, "no entry named %s", name);
  const auto held = f->locks.find(name);
  if (held != f->locks.end()) {
    *pinned_out = held->second.ptr;
    if (rung_out) *rung_out = held->second.rung;
    return NT_OK;
  }
  const Entry e = it->second;
  if (e.bytes == 0) return set_err(ctx, NT_ERR_INVALID_ARG, "entry %s is empty", name);
  const size_t n = size_t(up(e.bytes, kFileAlign));
  void* addr = f->base + e.off;
  Lock L;
  const bool in_place = g_refuse_in_place.load(std::memory_order_relaxed) == 0;
  // rung 0, "mmap pinned": the read-only shared mapping itself, registered read-only
  if (in_place && nt_host_register(ctx, addr, n, 1) == NT_OK) {
    L.rung = 0, L.ptr = addr;
  } else {
    // rung 1, "mmap pinned private": a private, writable, pre-faulted mapping of the range
    // (copy-on-write, so the file is never written), registered without the read-only flag
    const long pg = sysconf(_SC_PAGESIZE);
    const uint64_t page = pg > 0 ? uint64_t(pg) : kFileAlign;
    const uint64_t mbase = e.off / page * page;
    const size_t mlen = size_t(up(e.off - mbase + n, page));
    int flags = MAP_PRIVATE;
#ifdef MAP_POPULATE
    flags |= MAP_POPULATE;
#endif
    void* m = in_place ? mmap(nullptr, mlen, PROT_READ | PROT_WRITE, flags, f->fd, off_t(mbase)) : MAP_FAILED;
    if (m != MAP_FAILED) {
      void* p = static_cast<uint8_t*>(m) + (e.off - mbase);
      if (nt_host_register(ctx, p, n, 0) == NT_OK) {
        L.rung = 1, L.ptr = p, L.map = m, L.map_len = mlen;
      } else {
        munmap(m, mlen);
      }
    }
    if (!L.ptr) {
      if (!allow_copy)
        return set_err(ctx, NT_ERR_CUDA, "%s: the file's pages cannot be page-locked in place", name);
      // rung 2, "CPU memcpy": one CPU copy into page-locked memory
      int prev = -1;
      cudaGetDevice(&prev);
      if (prev != ctx->device) cudaSetDevice(ctx->device);
      void* h = nullptr;
      const cudaError_t ce = cudaHostAlloc(&h, n, cudaHostAllocPortable);
      if (prev >= 0 && prev != ctx->device) cudaSetDevice(prev);
      if (ce != cudaSuccess) {
        cudaGetLastError();
        return set_err(ctx, NT_ERR_OOM, "%s: page-locked copy of %zu bytes: %s", name, n, cudaGetErrorString(ce));
      }
      memcpy(h, addr, size_t(e.bytes));
      memset(static_cast<uint8_t*>(h) + e.bytes, 0, n - size_t(e.bytes));
      L.rung = 2, L.ptr = h;
    }
  }
  f->locks.emplace(name, L);
  *pinned_out = L.ptr;
  if (rung_out) *rung_out = L.rung;
  return NT_OK;
}

nt_status nt_debug_file_refuse_in_place(int on) {
  if (on != 0 && on != 1) return NT_ERR_INVALID_ARG;
  g_refuse_in_place.store(on);
  return NT_OK;
}

nt_status nt_file_unlock(nt_ctx* ctx, nt_file* f, const char* name) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  if (!f || !name) return set_err(ctx, NT_ERR_INVALID_ARG, "null pointer");
  const auto it = f->locks.find(name);
  if (it == f->locks.end()) return set_err(ctx, NT_ERR_INVALID_ARG, "entry %s is not page-locked", name);
  const Lock L = it->second;
  nt_status s = NT_OK;
  if (L.rung == 2) {
    const cudaError_t ce = cudaFreeHost(L.ptr);
    if (ce != cudaSuccess) {
      cudaGetLastError();
      s = set_err(ctx, NT_ERR_CUDA, "free page-locked copy of %s: %s", name, cudaGetErrorString(ce));
    }
  } else {
    s = nt_host_unregister(ctx, L.ptr);
    if (L.map) munmap(L.map, L.map_len);
  }
  f->locks.erase(it);  // released either way: a failed unregister leaves nothing to retry
  return s;
}

}  // extern "C"
