// st_index.cpp -- safetensors header parser, metadata-only index and views.
//
// "Disk tier safetensors streaming design audit (ComfyUI)":
//  - "FastSageTensors (fastsafetensors) capability audit": the header is parsed
//    into per-tensor dtype, shape and data_offsets with no tensor allocation;
//  - "Strategy summary (implemented)": a metadata-only index (TensorMeta /
//    SafeTensorIndex) whose keys/iteration never load tensors, and lazy
//    Prefix/Filter/Rename views;
//  - "Pipeline refactors": parameter counts and dtypes from metadata.
// The byte layout (8-byte little-endian N, N bytes of JSON, data section) is
// the format's public layout.
//
// The parser is a single pass over the header that validates JSON syntax
// (RFC 8259, nesting depth <= 64) while it decodes the schema directly into
// tensor records.  Schema/semantic defects are recorded in document order and
// reported only if the whole header is syntactically valid.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <memory>
#include <string>
#include <string_view>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "st_internal.h"
#include "st_index.h"

namespace stmat {

static thread_local std::string g_err;

st_status set_error(st_status s, const char *fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

static const char *const kDtypeNames[16] = {"BOOL", "U8",  "I8",  "I16", "U16", "I32",
                                            "U32",  "I64", "U64", "F16", "BF16", "F32",
                                            "F64",  "F8_E4M3", "F8_E5M2", "KEEP"};
static const uint8_t kDtypeSize[16] = {1, 1, 1, 2, 2, 4, 4, 8, 8, 2, 2, 4, 8, 1, 1, 0};

size_t dtype_size(int d) { return (d >= 0 && d < 16) ? kDtypeSize[d] : 0; }

static int dtype_from(std::string_view s) {
  for (int d = 0; d < 15; ++d)
    if (s == kDtypeNames[d]) return d;
  return -1;
}

namespace {

constexpr uint64_t kMaxHeader = 100000000ull;
constexpr int kMaxDepth = 64;

// ---------------------------------------------------------------- scanner

class Scanner {
 public:
  Scanner(const uint8_t *p, const uint8_t *e) : p_(p), e_(e) {}

  bool ok() const { return ok_; }
  bool at_end() { ws(); return p_ == e_; }
  bool peek(char c) { ws(); return p_ < e_ && *p_ == c; }
  bool eat(char c) {
    ws();
    if (p_ < e_ && *p_ == c) { ++p_; return true; }
    return false;
  }
  bool fail() { ok_ = false; return false; }
  // A mandatory character: its absence is a syntax error.
  bool expect(char c) { return eat(c) ? true : fail(); }

  void ws() {
    while (p_ < e_ && (*p_ == ' ' || *p_ == '\n' || *p_ == '\r' || *p_ == '\t')) ++p_;
  }

  // Value nesting: the top-level value is at depth 1.
  bool enter() { return ++depth_ <= kMaxDepth ? true : fail(); }
  void leave() { --depth_; }

  // JSON string -> UTF-8 bytes.  Rejects raw control characters, malformed
  // UTF-8, unpaired surrogates and U+0000.
  bool string(std::string *out) {
    ws();
    if (p_ >= e_ || *p_ != '"') return fail();
    ++p_;
    out->clear();
    const uint8_t *run = p_;
    while (true) {
      if (p_ >= e_) return fail();
      uint8_t c = *p_;
      if (c == '"') {
        out->append(reinterpret_cast<const char *>(run), p_ - run);
        ++p_;
        return true;
      }
      if (c < 0x20) return fail();
      if (c < 0x80 && c != '\\') { ++p_; continue; }
      if (c >= 0x80) {
        int k = utf8_seq(p_);
        if (!k) return fail();
        p_ += k;
        continue;
      }
      // escape
      out->append(reinterpret_cast<const char *>(run), p_ - run);
      if (e_ - p_ < 2) return fail();
      uint8_t x = p_[1];
      p_ += 2;
      switch (x) {
        case '"': out->push_back('"'); break;
        case '\\': out->push_back('\\'); break;
        case '/': out->push_back('/'); break;
        case 'b': out->push_back('\b'); break;
        case 'f': out->push_back('\f'); break;
        case 'n': out->push_back('\n'); break;
        case 'r': out->push_back('\r'); break;
        case 't': out->push_back('\t'); break;
        case 'u': {
          uint32_t cp;
          if (!hex4(&cp)) return fail();
          if (cp >= 0xDC00 && cp <= 0xDFFF) return fail();
          if (cp >= 0xD800 && cp <= 0xDBFF) {
            uint32_t lo;
            if (e_ - p_ < 2 || p_[0] != '\\' || p_[1] != 'u') return fail();
            p_ += 2;
            if (!hex4(&lo) || lo < 0xDC00 || lo > 0xDFFF) return fail();
            cp = 0x10000 + ((cp - 0xD800) << 10) + (lo - 0xDC00);
          }
          if (cp == 0) return fail();
          append_utf8(out, cp);
          break;
        }
        default: return fail();
      }
      run = p_;
    }
  }

  // Number token.  *plain: the token is digits only (a non-negative integer
  // written without sign, fraction or exponent); *value: its value if plain
  // and <= limit (else *plain is false).
  bool number(uint64_t limit, bool *plain, uint64_t *value) {
    ws();
    const uint8_t *s = p_;
    bool digits_only = true;
    if (p_ < e_ && *p_ == '-') { ++p_; digits_only = false; }
    if (p_ >= e_) return fail();
    if (*p_ == '0') {
      ++p_;
    } else if (*p_ >= '1' && *p_ <= '9') {
      while (p_ < e_ && *p_ >= '0' && *p_ <= '9') ++p_;
    } else {
      return fail();
    }
    const uint8_t *int_end = p_;
    if (p_ < e_ && *p_ == '.') {
      digits_only = false;
      ++p_;
      if (p_ >= e_ || *p_ < '0' || *p_ > '9') return fail();
      while (p_ < e_ && *p_ >= '0' && *p_ <= '9') ++p_;
    }
    if (p_ < e_ && (*p_ == 'e' || *p_ == 'E')) {
      digits_only = false;
      ++p_;
      if (p_ < e_ && (*p_ == '+' || *p_ == '-')) ++p_;
      if (p_ >= e_ || *p_ < '0' || *p_ > '9') return fail();
      while (p_ < e_ && *p_ >= '0' && *p_ <= '9') ++p_;
    }
    *plain = false;
    if (digits_only) {
      uint64_t v = 0;
      bool fits = true;
      for (const uint8_t *q = s; q < int_end; ++q) {
        uint64_t d = *q - '0';
        if (v > (limit - d) / 10) { fits = false; break; }
        v = v * 10 + d;
      }
      if (fits) { *plain = true; *value = v; }
    }
    return true;
  }

  bool literal(const char *lit) {
    ws();
    size_t n = strlen(lit);
    if (static_cast<size_t>(e_ - p_) < n || memcmp(p_, lit, n) != 0) return fail();
    p_ += n;
    return true;
  }

  // Any JSON value, validated and discarded.
  bool skip_value() {
    ws();
    if (p_ >= e_) return fail();
    if (!enter()) return false;
    bool r;
    switch (*p_) {
      case '{': {
        ++p_;
        r = true;
        if (eat('}')) break;
        std::string k;
        do {
          if (!string(&k) || !expect(':') || !skip_value()) { r = false; break; }
        } while (eat(','));
        if (r && !eat('}')) r = fail();
        break;
      }
      case '[': {
        ++p_;
        r = true;
        if (eat(']')) break;
        do {
          if (!skip_value()) { r = false; break; }
        } while (eat(','));
        if (r && !eat(']')) r = fail();
        break;
      }
      case '"': {
        std::string s;
        r = string(&s);
        break;
      }
      case 't': r = literal("true"); break;
      case 'f': r = literal("false"); break;
      case 'n': r = literal("null"); break;
      default: {
        bool plain;
        uint64_t v;
        r = number(0, &plain, &v);
      }
    }
    leave();
    return r;
  }

 private:
  bool hex4(uint32_t *out) {
    if (e_ - p_ < 4) return false;
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) {
      uint8_t c = p_[i];
      uint32_t d;
      if (c >= '0' && c <= '9') d = c - '0';
      else if (c >= 'a' && c <= 'f') d = c - 'a' + 10;
      else if (c >= 'A' && c <= 'F') d = c - 'A' + 10;
      else return false;
      v = (v << 4) | d;
    }
    p_ += 4;
    *out = v;
    return true;
  }

  // Length of the well-formed UTF-8 sequence at s (Unicode table 3-7), or 0.
  int utf8_seq(const uint8_t *s) const {
    uint8_t c = s[0];
    int n;
    uint8_t lo = 0x80, hi = 0xBF;
    if (c >= 0xC2 && c <= 0xDF) n = 2;
    else if (c == 0xE0) { n = 3; lo = 0xA0; }
    else if ((c >= 0xE1 && c <= 0xEC) || c == 0xEE || c == 0xEF) n = 3;
    else if (c == 0xED) { n = 3; hi = 0x9F; }
    else if (c == 0xF0) { n = 4; lo = 0x90; }
    else if (c >= 0xF1 && c <= 0xF3) n = 4;
    else if (c == 0xF4) { n = 4; hi = 0x8F; }
    else return 0;
    if (e_ - s < n) return 0;
    if (s[1] < lo || s[1] > hi) return 0;
    for (int i = 2; i < n; ++i)
      if (s[i] < 0x80 || s[i] > 0xBF) return 0;
    return n;
  }

  static void append_utf8(std::string *o, uint32_t cp) {
    if (cp < 0x80) {
      o->push_back(static_cast<char>(cp));
    } else if (cp < 0x800) {
      o->push_back(static_cast<char>(0xC0 | (cp >> 6)));
      o->push_back(static_cast<char>(0x80 | (cp & 0x3F)));
    } else if (cp < 0x10000) {
      o->push_back(static_cast<char>(0xE0 | (cp >> 12)));
      o->push_back(static_cast<char>(0x80 | ((cp >> 6) & 0x3F)));
      o->push_back(static_cast<char>(0x80 | (cp & 0x3F)));
    } else {
      o->push_back(static_cast<char>(0xF0 | (cp >> 18)));
      o->push_back(static_cast<char>(0x80 | ((cp >> 12) & 0x3F)));
      o->push_back(static_cast<char>(0x80 | ((cp >> 6) & 0x3F)));
      o->push_back(static_cast<char>(0x80 | (cp & 0x3F)));
    }
  }

  const uint8_t *p_, *e_;
  int depth_ = 0;
  bool ok_ = true;
};

// First schema/semantic defect in document order.
struct Defect {
  st_status status = ST_OK;
  std::string msg;
  void note(st_status s, std::string m) {
    if (status == ST_OK) { status = s; msg = std::move(m); }
  }
};

// Parses one tensor entry object; returns the entry's status.
st_status parse_entry(Scanner &sc, const std::string &name, uint64_t data_bytes, Tensor *t,
                      std::string *why) {
  bool struct_bad = false, shape_bad = false, off_bad = false;
  bool seen_dtype = false, seen_shape = false, seen_off = false;
  int dtype = -2;  // -2: not a string, -1: unknown name
  size_t n_off = 0;
  uint64_t off[2] = {0, 0};
  std::vector<int64_t> dims;
  std::string key, sval;
  if (!sc.peek('{')) {
    if (!sc.skip_value()) return ST_OK;
    *why = "entry is not an object";
    return ST_E_HEADER_JSON;
  }
  if (!sc.enter()) return ST_OK;
  sc.eat('{');
  if (!sc.eat('}')) {
    do {
      if (!sc.string(&key) || !sc.expect(':')) return ST_OK;
      int which = key == "dtype" ? 0 : key == "shape" ? 1 : key == "data_offsets" ? 2 : 3;
      bool *seen = which == 0 ? &seen_dtype : which == 1 ? &seen_shape : which == 2 ? &seen_off : nullptr;
      if (which == 3 || *seen) {
        struct_bad = true;
        if (!sc.skip_value()) return ST_OK;
        continue;
      }
      *seen = true;
      if (which == 0) {
        if (sc.peek('"')) {
          if (!sc.enter()) return ST_OK;
          if (!sc.string(&sval)) return ST_OK;
          sc.leave();
          dtype = dtype_from(sval);
        } else {
          struct_bad = true;
          if (!sc.skip_value()) return ST_OK;
        }
      } else {
        if (!sc.peek('[')) {
          struct_bad = true;
          if (!sc.skip_value()) return ST_OK;
          continue;
        }
        if (!sc.enter()) return ST_OK;
        sc.eat('[');
        size_t count = 0;
        if (!sc.eat(']')) {
          do {
            sc.ws();
            if (sc.peek('{') || sc.peek('[') || sc.peek('"') || sc.peek('t') || sc.peek('f') ||
                sc.peek('n')) {
              struct_bad = true;
              if (!sc.skip_value()) return ST_OK;
            } else {
              if (!sc.enter()) return ST_OK;
              bool plain;
              uint64_t v = 0;
              if (!sc.number(which == 1 ? static_cast<uint64_t>(INT64_MAX) : UINT64_MAX, &plain, &v))
                return ST_OK;
              sc.leave();
              if (which == 1) {
                if (!plain) shape_bad = true;
                dims.push_back(static_cast<int64_t>(v));
              } else {
                if (!plain) off_bad = true;
                if (count < 2) off[count] = v;
              }
            }
            ++count;
          } while (sc.eat(','));
          if (!sc.eat(']')) return sc.fail(), ST_OK;
        }
        sc.leave();
        if (which == 2) n_off = count;
      }
    } while (sc.eat(','));
    if (!sc.eat('}')) return sc.fail(), ST_OK;
  }
  sc.leave();
  // Checks in order: schema, dtype, shape, offsets.
  if (struct_bad || !seen_dtype || !seen_shape || !seen_off || dtype == -2 || n_off != 2) {
    *why = "entry must have exactly dtype (string), shape (array of numbers) and data_offsets (two numbers)";
    return ST_E_HEADER_JSON;
  }
  if (dtype < 0) {
    *why = "unknown dtype \"" + sval + "\"";
    return ST_E_DTYPE;
  }
  uint64_t numel = 1;
  if (shape_bad) {
    *why = "shape dimensions must be non-negative integers <= 2^63-1";
    return ST_E_SHAPE;
  }
  for (int64_t d : dims) {
    uint64_t u = static_cast<uint64_t>(d);
    if (u != 0 && numel > UINT64_MAX / u) {
      *why = "shape product overflows 64 bits";
      return ST_E_SHAPE;
    }
    numel *= u;
  }
  uint64_t isz = kDtypeSize[dtype];
  if (numel > UINT64_MAX / isz) {
    *why = "tensor byte size overflows 64 bits";
    return ST_E_SHAPE;
  }
  uint64_t nbytes = numel * isz;
  if (off_bad) {
    *why = "data_offsets must be non-negative integers < 2^64";
    return ST_E_OFFSETS;
  }
  if (off[0] > off[1] || off[1] > data_bytes || off[1] - off[0] != nbytes) {
    char b[256];
    snprintf(b, sizeof b,
             "data_offsets [%llu, %llu] do not hold %llu bytes inside a %llu-byte data section",
             (unsigned long long)off[0], (unsigned long long)off[1], (unsigned long long)nbytes,
             (unsigned long long)data_bytes);
    *why = b;
    return ST_E_OFFSETS;
  }
  t->name = name;
  t->dtype = dtype;
  t->shape = std::move(dims);
  t->numel = numel;
  t->begin = off[0];
  t->end = off[1];
  return ST_OK;
}

// "__metadata__": an object of strings with unique keys.
st_status parse_metadata(Scanner &sc, std::vector<std::pair<std::string, std::string>> *meta) {
  if (!sc.peek('{')) return sc.skip_value() ? ST_E_HEADER_JSON : ST_OK;
  if (!sc.enter()) return ST_OK;
  sc.eat('{');
  bool bad = false;
  std::unordered_set<std::string> keys;
  std::string k, v;
  if (!sc.eat('}')) {
    do {
      if (!sc.string(&k) || !sc.expect(':')) return ST_OK;
      if (!keys.insert(k).second) bad = true;
      if (sc.peek('"')) {
        if (!sc.enter() || !sc.string(&v)) return ST_OK;
        sc.leave();
        meta->emplace_back(k, v);
      } else {
        bad = true;
        if (!sc.skip_value()) return ST_OK;
      }
    } while (sc.eat(','));
    if (!sc.eat('}')) return sc.fail(), ST_OK;
  }
  sc.leave();
  return bad ? ST_E_HEADER_JSON : ST_OK;
}

}  // namespace

// Parses the JSON of one header (n bytes) for a data section of data_bytes.
st_status parse_header(const uint8_t *json, size_t n, uint64_t data_bytes, Core *core) {
  Scanner sc(json, json + n);
  Defect defect;
  std::unordered_set<std::string> seen;
  std::string name;
  bool top_is_object = sc.peek('{');
  if (!top_is_object) {
    sc.skip_value();
    if (sc.ok() && !sc.at_end()) sc.fail();
    return set_error(ST_E_HEADER_JSON, "header is not a JSON object");
  }
  sc.enter();
  sc.eat('{');
  if (!sc.eat('}')) {
    do {
      if (!sc.string(&name) || !sc.expect(':')) break;
      bool fresh = seen.insert(name).second;
      if (!fresh) defect.note(ST_E_DUP_KEY, "name \"" + name + "\" appears twice");
      if (name == "__metadata__") {
        std::vector<std::pair<std::string, std::string>> meta;
        st_status s = parse_metadata(sc, &meta);
        if (!sc.ok()) break;
        if (s != ST_OK) defect.note(s, "__metadata__ must be an object of strings with unique keys");
        if (fresh && s == ST_OK) core->meta = std::move(meta);
      } else {
        Tensor t;
        std::string why;
        st_status s = parse_entry(sc, name, data_bytes, &t, &why);
        if (!sc.ok()) break;
        if (s != ST_OK) defect.note(s, "tensor \"" + name + "\": " + why);
        else if (fresh) core->tensors.push_back(std::move(t));
      }
    } while (sc.eat(','));
    if (sc.ok() && !sc.eat('}')) sc.fail();
  }
  sc.leave();
  if (sc.ok() && !sc.at_end()) sc.fail();
  if (!sc.ok()) return set_error(ST_E_HEADER_JSON, "header is not valid JSON (RFC 8259, depth <= 64)");
  if (defect.status != ST_OK) return set_error(defect.status, "%s", defect.msg.c_str());
  // Index order and tiling of the data section.
  std::vector<Tensor> &ts = core->tensors;
  std::sort(ts.begin(), ts.end(), [](const Tensor &a, const Tensor &b) {
    if (a.begin != b.begin) return a.begin < b.begin;
    if (a.end != b.end) return a.end < b.end;
    return a.name < b.name;
  });
  uint64_t at = 0;
  for (const Tensor &t : ts) {
    if (t.begin != at)
      return set_error(ST_E_OFFSETS, "tensor \"%s\" starts at %llu but the previous range ends at %llu (%s)",
                       t.name.c_str(), (unsigned long long)t.begin, (unsigned long long)at,
                       t.begin > at ? "hole" : "overlap");
    at = t.end;
  }
  if (at != data_bytes)
    return set_error(ST_E_OFFSETS, "tensors cover %llu of %llu data bytes", (unsigned long long)at,
                     (unsigned long long)data_bytes);
  core->data_bytes = data_bytes;
  return ST_OK;
}

std::shared_ptr<IndexData> make_root(std::shared_ptr<const Core> core) {
  auto d = std::make_shared<IndexData>();
  d->core = core;
  d->ent.resize(core->tensors.size());
  d->names.resize(core->tensors.size());
  for (size_t i = 0; i < core->tensors.size(); ++i) {
    d->ent[i] = static_cast<uint32_t>(i);
    d->names[i] = core->tensors[i].name.c_str();
  }
  return d;
}

st_status finish_view(IndexData *d) {
  d->pos.reserve(d->names.size() * 2);
  for (size_t i = 0; i < d->names.size(); ++i)
    if (!d->pos.emplace(std::string_view(d->names[i]), static_cast<uint32_t>(i)).second)
      return set_error(ST_E_DUP_KEY, "two tensors are named \"%s\" in the view", d->names[i]);
  return ST_OK;
}

}  // namespace stmat

using namespace stmat;

struct st_index {
  std::shared_ptr<const IndexData> d;
};

namespace stmat {
const IndexData *index_data(const st_index *ix) { return ix->d.get(); }
std::shared_ptr<const IndexData> index_ref(const st_index *ix) { return ix->d; }
}  // namespace stmat

static st_status wrap(std::shared_ptr<IndexData> d, st_index **out) {
  st_status s = finish_view(d.get());
  if (s != ST_OK) return s;
  st_index *ix = new (std::nothrow) st_index;
  if (!ix) return set_error(ST_E_NOMEM, "out of host memory");
  ix->d = std::move(d);
  *out = ix;
  return ST_OK;
}

extern "C" {

const char *st_last_error(void) { return g_err.c_str(); }

const char *st_status_name(st_status s) {
  static const char *const n[] = {"ST_OK",       "ST_E_INVAL",    "ST_E_TRUNCATED", "ST_E_HEADER_JSON",
                                  "ST_E_HEADER_TOO_LARGE", "ST_E_DUP_KEY", "ST_E_DTYPE", "ST_E_SHAPE",
                                  "ST_E_OFFSETS", "ST_E_NOT_FOUND", "ST_E_UNSUPPORTED_CAST",
                                  "ST_E_ALIGN",  "ST_E_NOMEM",    "ST_E_CUDA",      "ST_E_DEVICE", "ST_E_IO"};
  return (s >= 0 && s <= ST_E_IO) ? n[s] : "ST_E_UNKNOWN";
}

size_t st_dtype_size(st_dtype d) { return dtype_size(d); }
const char *st_dtype_name(st_dtype d) { return (d >= 0 && d < 16) ? kDtypeNames[d] : nullptr; }
uint32_t st_version(void) { return 0x000100; }

st_status st_header_size(const uint8_t *first8, size_t len, uint64_t *header_len) {
  if (!header_len || (len && !first8)) return set_error(ST_E_INVAL, "NULL argument");
  if (len < 8) return set_error(ST_E_TRUNCATED, "%zu bytes given, the length prefix needs 8", len);
  uint64_t n = 0;
  for (int i = 7; i >= 0; --i) n = (n << 8) | first8[i];
  if (n > kMaxHeader)
    return set_error(ST_E_HEADER_TOO_LARGE, "header length %llu exceeds %llu", (unsigned long long)n,
                     (unsigned long long)kMaxHeader);
  *header_len = n;
  return ST_OK;
}

st_status st_index_build(const uint8_t *header_bytes, size_t len, uint64_t data_bytes, st_index **out) {
  if (!out) return set_error(ST_E_INVAL, "NULL out");
  *out = nullptr;
  uint64_t n;
  st_status s = st_header_size(header_bytes, len, &n);
  if (s != ST_OK) return s;
  if (n > len - 8)
    return set_error(ST_E_TRUNCATED, "header needs %llu bytes after the prefix, %zu given",
                     (unsigned long long)n, len - 8);
  auto core = std::make_shared<Core>();
  core->header_len = n;
  try {
    s = parse_header(header_bytes + 8, n, data_bytes, core.get());
    if (s != ST_OK) return s;
    return wrap(make_root(core), out);
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory while parsing the header");
  }
}

st_status st_index_build_file(const uint8_t *file, uint64_t file_len, st_index **out) {
  if (!out) return set_error(ST_E_INVAL, "NULL out");
  *out = nullptr;
  uint64_t n;
  st_status s = st_header_size(file, file_len, &n);
  if (s != ST_OK) return s;
  if (n > file_len - 8)
    return set_error(ST_E_TRUNCATED, "header length %llu exceeds the %llu bytes after the prefix",
                     (unsigned long long)n, (unsigned long long)(file_len - 8));
  return st_index_build(file, 8 + n, file_len - 8 - n, out);
}

void st_index_free(st_index *ix) { delete ix; }

st_status st_index_count(const st_index *ix, size_t *count) {
  if (!ix || !count) return set_error(ST_E_INVAL, "NULL argument");
  *count = ix->d->ent.size();
  return ST_OK;
}

st_status st_index_get(const st_index *ix, size_t i, st_tensor_info *info) {
  if (!ix || !info) return set_error(ST_E_INVAL, "NULL argument");
  if (i >= ix->d->ent.size()) return set_error(ST_E_INVAL, "index %zu out of range", i);
  const Tensor &t = ix->d->core->tensors[ix->d->ent[i]];
  info->name = ix->d->names[i];
  info->dtype = static_cast<st_dtype>(t.dtype);
  info->ndim = static_cast<int32_t>(t.shape.size());
  info->shape = t.shape.data();
  info->numel = t.numel;
  info->begin = t.begin;
  info->end = t.end;
  return ST_OK;
}

st_status st_index_find(const st_index *ix, const char *name, size_t *i) {
  if (!ix || !name || !i) return set_error(ST_E_INVAL, "NULL argument");
  auto it = ix->d->pos.find(std::string_view(name));
  if (it == ix->d->pos.end()) return set_error(ST_E_NOT_FOUND, "no tensor named \"%s\"", name);
  *i = it->second;
  return ST_OK;
}

st_status st_index_sizes(const st_index *ix, uint64_t *header_len, uint64_t *data_bytes) {
  if (!ix) return set_error(ST_E_INVAL, "NULL index");
  if (header_len) *header_len = ix->d->core->header_len;
  if (data_bytes) *data_bytes = ix->d->core->data_bytes;
  return ST_OK;
}

st_status st_index_numel(const st_index *ix, uint64_t *total, uint64_t *counts) {
  if (!ix) return set_error(ST_E_INVAL, "NULL index");
  uint64_t sum = 0, c[15] = {0};
  for (uint32_t e : ix->d->ent) {
    const Tensor &t = ix->d->core->tensors[e];
    sum += t.numel;
    c[t.dtype] += t.numel;
  }
  if (total) *total = sum;
  if (counts) memcpy(counts, c, sizeof c);
  return ST_OK;
}

st_status st_index_metadata_count(const st_index *ix, size_t *count) {
  if (!ix || !count) return set_error(ST_E_INVAL, "NULL argument");
  *count = ix->d->core->meta.size();
  return ST_OK;
}

st_status st_index_metadata_get(const st_index *ix, size_t i, const char **key, const char **value) {
  if (!ix || !key || !value) return set_error(ST_E_INVAL, "NULL argument");
  if (i >= ix->d->core->meta.size()) return set_error(ST_E_INVAL, "metadata index %zu out of range", i);
  *key = ix->d->core->meta[i].first.c_str();
  *value = ix->d->core->meta[i].second.c_str();
  return ST_OK;
}

st_status st_view_prefix(const st_index *parent, const char *prefix, st_index **out) {
  if (!parent || !prefix || !out) return set_error(ST_E_INVAL, "NULL argument");
  *out = nullptr;
  try {
    auto d = std::make_shared<IndexData>();
    d->core = parent->d->core;
    d->parent = parent->d;
    size_t k = strlen(prefix);
    for (size_t i = 0; i < parent->d->ent.size(); ++i) {
      const char *nm = parent->d->names[i];
      if (strncmp(nm, prefix, k) == 0) {
        d->ent.push_back(parent->d->ent[i]);
        d->names.push_back(nm + k);
      }
    }
    return wrap(std::move(d), out);
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory");
  }
}

st_status st_view_filter(const st_index *parent, const char *const *names, size_t n, st_index **out) {
  if (!parent || (n && !names) || !out) return set_error(ST_E_INVAL, "NULL argument");
  *out = nullptr;
  try {
    std::vector<char> keep(parent->d->ent.size(), 0);
    for (size_t j = 0; j < n; ++j) {
      if (!names[j]) return set_error(ST_E_INVAL, "NULL name at %zu", j);
      auto it = parent->d->pos.find(std::string_view(names[j]));
      if (it == parent->d->pos.end()) return set_error(ST_E_NOT_FOUND, "no tensor named \"%s\"", names[j]);
      keep[it->second] = 1;
    }
    auto d = std::make_shared<IndexData>();
    d->core = parent->d->core;
    d->parent = parent->d;
    for (size_t i = 0; i < keep.size(); ++i)
      if (keep[i]) {
        d->ent.push_back(parent->d->ent[i]);
        d->names.push_back(parent->d->names[i]);
      }
    return wrap(std::move(d), out);
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory");
  }
}

st_status st_view_rename(const st_index *parent, const char *const *from, const char *const *to, size_t n,
                         st_index **out) {
  if (!parent || (n && (!from || !to)) || !out) return set_error(ST_E_INVAL, "NULL argument");
  *out = nullptr;
  for (size_t j = 0; j < n; ++j)
    if (!from[j] || !to[j]) return set_error(ST_E_INVAL, "NULL rule at %zu", j);
  try {
    auto d = std::make_shared<IndexData>();
    d->core = parent->d->core;
    d->parent = parent->d;
    std::vector<size_t> flen(n);
    for (size_t j = 0; j < n; ++j) flen[j] = strlen(from[j]);
    for (size_t i = 0; i < parent->d->ent.size(); ++i) {
      const char *nm = parent->d->names[i];
      const char *res = nm;
      for (size_t j = 0; j < n; ++j)
        if (strncmp(nm, from[j], flen[j]) == 0) {
          d->owned.emplace_back(std::string(to[j]) + (nm + flen[j]));
          res = d->owned.back().c_str();
          break;
        }
      d->ent.push_back(parent->d->ent[i]);
      d->names.push_back(res);
    }
    return wrap(std::move(d), out);
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory");
  }
}

}  // extern "C"

extern "C" {

st_status st_index_concat(const st_index *const *parts, size_t n, uint64_t align, uint64_t *bases, st_index **out) {
  if (!parts || !n || !bases || !out) return set_error(ST_E_INVAL, "NULL argument or no parts");
  *out = nullptr;
  if (align == 0 || (align & (align - 1))) return set_error(ST_E_INVAL, "align %llu is not a power of two",
                                                            (unsigned long long)align);
  for (size_t k = 0; k < n; ++k)
    if (!parts[k]) return set_error(ST_E_INVAL, "NULL part %zu", k);
  try {
    auto core = std::make_shared<Core>();
    uint64_t at = 0;
    for (size_t k = 0; k < n; ++k) {
      const IndexData &p = *parts[k]->d;
      const uint64_t size = p.core->data_bytes;
      const uint64_t base = (at + align - 1) & ~(align - 1);
      if (base < at || base + size < base) return set_error(ST_E_OFFSETS, "the joined data sections overflow 64 bits");
      bases[k] = base;
      at = base + size;
      for (size_t i = 0; i < p.ent.size(); ++i) {
        Tensor t = p.core->tensors[p.ent[i]];
        t.name = p.names[i];
        t.begin += base;
        t.end += base;
        core->tensors.push_back(std::move(t));
      }
      for (const auto &kv : p.core->meta) {
        bool seen = false;
        for (const auto &m : core->meta) seen = seen || m.first == kv.first;
        if (!seen) core->meta.push_back(kv);
      }
    }
    core->data_bytes = at;
    return wrap(make_root(core), out);
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory");
  }
}

}  // extern "C"
