/*
 * stmat_oracle.c -- plain, slow, single-threaded CPU oracle for safetensors
 * materialization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (sources):
 *  - "Disk tier safetensors streaming design audit (ComfyUI)", section
 *    "FastSageTensors (fastsafetensors) capability audit": the header is parsed
 *    into per-tensor dtype, shape and data_offsets without allocating tensors.
 *    The byte layout itself is not printed on the pages; the reading taken is
 *    the public safetensors layout: an unsigned 64-bit little-endian header
 *    length N, N bytes of UTF-8 JSON, then the data section, with
 *    data_offsets = [begin, end) relative to the data section's first byte.
 *  - Same page, "Strategy summary (implemented)", "Streaming safetensors
 *    mapping": metadata-only index plus Prefix/Filter/Rename views.
 *  - Same page, "ComfyUI load path + eager materialization sites": the
 *    scaled-FP8 conversion in comfy/sd.py; and "VRAM/RAM offload logic":
 *    weight casting (comfy_cast_weights).  Reading: an fp8 weight is decoded
 *    exactly, multiplied by its per-tensor fp32 scale with one IEEE binary32
 *    multiply, then rounded to the target with round-to-nearest-even.
 *
 * Every float conversion is written from the format definitions:
 *  - IEEE 754 binary32 / binary16 and bfloat16 (binary32's upper 16 bits);
 *  - OCP 8-bit floating point (OFP8): E4M3 (bias 7, no infinities, only
 *    S.1111.111 is NaN, max 448) and E5M2 (bias 15, IEEE-like specials).
 * Decoding produces the exact value as a double (every value of these formats
 * is a double); encoding rounds an exact double to the nearest representable
 * value, ties to even, with gradual underflow and overflow to infinity.  Any
 * NaN result becomes the target's positive quiet NaN (bf16 0x7FC0, f16 0x7E00,
 * f32 0x7FC00000).  Integer and bool tensors, and tensors whose target equals
 * their own dtype, are copied byte for byte.
 *
 * Build: gcc -O1 -std=c11 -fPIC -shared -ffp-contract=off (no fast-math): the
 * one binary32 multiply must stay a single IEEE multiply.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes (the C ABI's numbering, restated here on purpose). */
enum {
  OR_OK = 0,
  OR_E_INVAL = 1,
  OR_E_TRUNCATED = 2,
  OR_E_HEADER_JSON = 3,
  OR_E_HEADER_TOO_LARGE = 4,
  OR_E_DUP_KEY = 5,
  OR_E_DTYPE = 6,
  OR_E_SHAPE = 7,
  OR_E_OFFSETS = 8,
  OR_E_NOT_FOUND = 9,
  OR_E_UNSUPPORTED_CAST = 10,
  OR_E_ALIGN = 11,
  OR_E_NOMEM = 12
};

/* Dtype codes, in the C ABI's numbering. */
enum {
  OR_BOOL = 0, OR_U8, OR_I8, OR_I16, OR_U16, OR_I32, OR_U32, OR_I64, OR_U64,
  OR_F16, OR_BF16, OR_F32, OR_F64, OR_F8_E4M3, OR_F8_E5M2, OR_KEEP
};

static const char *const kNames[15] = {
    "BOOL", "U8",  "I8",  "I16", "U16", "I32",     "U32",    "I64",
    "U64",  "F16", "BF16", "F32", "F64", "F8_E4M3", "F8_E5M2"};
static const int kSize[15] = {1, 1, 1, 2, 2, 4, 4, 8, 8, 2, 2, 4, 8, 1, 1};

#define OR_MAX_HEADER 100000000ull /* the format's customary 100 MB cap */

int or_itemsize(int dtype) { return (dtype >= 0 && dtype < 15) ? kSize[dtype] : 0; }

/* ===================================================================== */
/* 1. A small generic JSON reader (RFC 8259) producing a value tree.      */
/* ===================================================================== */

typedef enum { J_NULL, J_TRUE, J_FALSE, J_NUM, J_STR, J_ARR, J_OBJ } jkind;

typedef struct jval {
  jkind kind;
  char *text;          /* J_STR: decoded bytes, NUL-terminated; J_NUM: raw token */
  size_t n;            /* J_ARR / J_OBJ: number of members */
  struct jval *items;  /* member values */
  char **keys;         /* J_OBJ: decoded keys */
} jval;

typedef struct {
  const uint8_t *p;
  const uint8_t *end;
  int depth;
} jreader;

static void jfree(jval *v) {
  size_t i;
  if (!v) return;
  free(v->text);
  for (i = 0; i < v->n; i++) {
    jfree(&v->items[i]);
    if (v->keys) free(v->keys[i]);
  }
  free(v->items);
  free(v->keys);
  memset(v, 0, sizeof(*v));
}

static void jskip_ws(jreader *r) {
  while (r->p < r->end && (*r->p == ' ' || *r->p == '\t' || *r->p == '\n' || *r->p == '\r')) r->p++;
}

/* Append one code point as UTF-8. */
static void put_utf8(char *out, size_t *len, uint32_t cp) {
  if (cp < 0x80) {
    out[(*len)++] = (char)cp;
  } else if (cp < 0x800) {
    out[(*len)++] = (char)(0xC0 | (cp >> 6));
    out[(*len)++] = (char)(0x80 | (cp & 0x3F));
  } else if (cp < 0x10000) {
    out[(*len)++] = (char)(0xE0 | (cp >> 12));
    out[(*len)++] = (char)(0x80 | ((cp >> 6) & 0x3F));
    out[(*len)++] = (char)(0x80 | (cp & 0x3F));
  } else {
    out[(*len)++] = (char)(0xF0 | (cp >> 18));
    out[(*len)++] = (char)(0x80 | ((cp >> 12) & 0x3F));
    out[(*len)++] = (char)(0x80 | ((cp >> 6) & 0x3F));
    out[(*len)++] = (char)(0x80 | (cp & 0x3F));
  }
}

static int hex4(const uint8_t *s, uint32_t *out) {
  uint32_t v = 0;
  int i;
  for (i = 0; i < 4; i++) {
    int c = s[i], d;
    if (c >= '0' && c <= '9') d = c - '0';
    else if (c >= 'a' && c <= 'f') d = c - 'a' + 10;
    else if (c >= 'A' && c <= 'F') d = c - 'A' + 10;
    else return 0;
    v = v * 16 + (uint32_t)d;
  }
  *out = v;
  return 1;
}

/* Length of one well-formed UTF-8 sequence starting at s (Unicode 15, table 3-7),
   or 0 if it is not well formed. */
static int utf8_len(const uint8_t *s, const uint8_t *end) {
  uint8_t c = s[0];
  int need, i;
  uint8_t lo = 0x80, hi = 0xBF;
  if (c < 0x80) return 1;
  if (c >= 0xC2 && c <= 0xDF) need = 1;
  else if (c == 0xE0) { need = 2; lo = 0xA0; }
  else if (c >= 0xE1 && c <= 0xEC) need = 2;
  else if (c == 0xED) { need = 2; hi = 0x9F; }
  else if (c >= 0xEE && c <= 0xEF) need = 2;
  else if (c == 0xF0) { need = 3; lo = 0x90; }
  else if (c >= 0xF1 && c <= 0xF3) need = 3;
  else if (c == 0xF4) { need = 3; hi = 0x8F; }
  else return 0;
  if (end - s < need + 1) return 0;
  for (i = 1; i <= need; i++) {
    uint8_t b = s[i];
    uint8_t l = (i == 1) ? lo : 0x80, h = (i == 1) ? hi : 0xBF;
    if (b < l || b > h) return 0;
  }
  return need + 1;
}

/* Reads a JSON string (the opening quote is at r->p).  Rejects raw control
   characters, malformed UTF-8, lone surrogates and U+0000 (names are C strings). */
static int jread_string(jreader *r, char **out) {
  const uint8_t *s = r->p + 1;
  size_t cap = 16, len = 0;
  char *buf;
  if (r->p >= r->end || *r->p != '"') return 0;
  buf = (char *)malloc(cap);
  if (!buf) return 0;
  while (1) {
    uint8_t c;
    if (len + 8 >= cap) {
      char *nb;
      cap *= 2;
      nb = (char *)realloc(buf, cap);
      if (!nb) { free(buf); return 0; }
      buf = nb;
    }
    if (s >= r->end) { free(buf); return 0; }
    c = *s;
    if (c == '"') { s++; break; }
    if (c < 0x20) { free(buf); return 0; }
    if (c == '\\') {
      uint32_t cp;
      if (s + 1 >= r->end) { free(buf); return 0; }
      c = s[1];
      s += 2;
      switch (c) {
        case '"': buf[len++] = '"'; break;
        case '\\': buf[len++] = '\\'; break;
        case '/': buf[len++] = '/'; break;
        case 'b': buf[len++] = '\b'; break;
        case 'f': buf[len++] = '\f'; break;
        case 'n': buf[len++] = '\n'; break;
        case 'r': buf[len++] = '\r'; break;
        case 't': buf[len++] = '\t'; break;
        case 'u':
          if (r->end - s < 4 || !hex4(s, &cp)) { free(buf); return 0; }
          s += 4;
          if (cp >= 0xD800 && cp <= 0xDBFF) { /* needs a low surrogate next */
            uint32_t lo;
            if (r->end - s < 6 || s[0] != '\\' || s[1] != 'u' || !hex4(s + 2, &lo) ||
                lo < 0xDC00 || lo > 0xDFFF) { free(buf); return 0; }
            s += 6;
            cp = 0x10000 + ((cp - 0xD800) << 10) + (lo - 0xDC00);
          } else if (cp >= 0xDC00 && cp <= 0xDFFF) {
            free(buf); return 0;
          }
          if (cp == 0) { free(buf); return 0; }
          put_utf8(buf, &len, cp);
          break;
        default: free(buf); return 0;
      }
      continue;
    }
    {
      int k = utf8_len(s, r->end), i;
      if (k == 0) { free(buf); return 0; }
      for (i = 0; i < k; i++) buf[len++] = (char)s[i];
      s += k;
    }
  }
  buf[len] = 0;
  r->p = s;
  *out = buf;
  return 1;
}

static int jread_value(jreader *r, jval *v);

static int jread_number(jreader *r, jval *v) {
  const uint8_t *s = r->p, *start = r->p;
  size_t len;
  if (s < r->end && *s == '-') s++;
  if (s >= r->end) return 0;
  if (*s == '0') s++;
  else if (*s >= '1' && *s <= '9') { while (s < r->end && *s >= '0' && *s <= '9') s++; }
  else return 0;
  if (s < r->end && *s == '.') {
    s++;
    if (s >= r->end || !(*s >= '0' && *s <= '9')) return 0;
    while (s < r->end && *s >= '0' && *s <= '9') s++;
  }
  if (s < r->end && (*s == 'e' || *s == 'E')) {
    s++;
    if (s < r->end && (*s == '+' || *s == '-')) s++;
    if (s >= r->end || !(*s >= '0' && *s <= '9')) return 0;
    while (s < r->end && *s >= '0' && *s <= '9') s++;
  }
  len = (size_t)(s - start);
  v->kind = J_NUM;
  v->text = (char *)malloc(len + 1);
  if (!v->text) return 0;
  memcpy(v->text, start, len);
  v->text[len] = 0;
  r->p = s;
  return 1;
}

static int jlit(jreader *r, const char *lit) {
  size_t n = strlen(lit);
  if ((size_t)(r->end - r->p) < n || memcmp(r->p, lit, n) != 0) return 0;
  r->p += n;
  return 1;
}

/* Appends one member to an array/object under construction. */
static int jpush(jval *v, size_t *cap, char *key) {
  if (v->n == *cap) {
    size_t nc = *cap ? *cap * 2 : 4;
    jval *ni = (jval *)realloc(v->items, nc * sizeof(jval));
    if (!ni) return 0;
    v->items = ni;
    if (v->kind == J_OBJ) {
      char **nk = (char **)realloc(v->keys, nc * sizeof(char *));
      if (!nk) return 0;
      v->keys = nk;
    }
    *cap = nc;
  }
  memset(&v->items[v->n], 0, sizeof(jval));
  if (v->kind == J_OBJ) v->keys[v->n] = key;
  v->n++;
  return 1;
}

static int jread_value(jreader *r, jval *v) {
  memset(v, 0, sizeof(*v));
  jskip_ws(r);
  if (r->p >= r->end) return 0;
  if (++r->depth > 64) return 0; /* nesting limit */
  switch (*r->p) {
    case '{': {
      size_t cap = 0;
      v->kind = J_OBJ;
      r->p++;
      jskip_ws(r);
      if (r->p < r->end && *r->p == '}') { r->p++; break; }
      while (1) {
        char *key = NULL;
        jskip_ws(r);
        if (!jread_string(r, &key)) return 0;
        if (!jpush(v, &cap, key)) { free(key); return 0; }
        jskip_ws(r);
        if (r->p >= r->end || *r->p != ':') return 0;
        r->p++;
        if (!jread_value(r, &v->items[v->n - 1])) return 0;
        jskip_ws(r);
        if (r->p < r->end && *r->p == ',') { r->p++; continue; }
        if (r->p < r->end && *r->p == '}') { r->p++; break; }
        return 0;
      }
      break;
    }
    case '[': {
      size_t cap = 0;
      v->kind = J_ARR;
      r->p++;
      jskip_ws(r);
      if (r->p < r->end && *r->p == ']') { r->p++; break; }
      while (1) {
        if (!jpush(v, &cap, NULL)) return 0;
        if (!jread_value(r, &v->items[v->n - 1])) return 0;
        jskip_ws(r);
        if (r->p < r->end && *r->p == ',') { r->p++; continue; }
        if (r->p < r->end && *r->p == ']') { r->p++; break; }
        return 0;
      }
      break;
    }
    case '"':
      v->kind = J_STR;
      if (!jread_string(r, &v->text)) return 0;
      break;
    case 't': v->kind = J_TRUE; if (!jlit(r, "true")) return 0; break;
    case 'f': v->kind = J_FALSE; if (!jlit(r, "false")) return 0; break;
    case 'n': v->kind = J_NULL; if (!jlit(r, "null")) return 0; break;
    default:
      if (!jread_number(r, v)) return 0;
  }
  r->depth--;
  return 1;
}

/* A JSON number token that is a non-negative integer (digits only) and at most
   `limit`.  Returns 1 and the value, or 0. */
static int jnum_to_u64(const jval *v, uint64_t limit, uint64_t *out) {
  const char *s;
  uint64_t x = 0;
  if (v->kind != J_NUM) return 0;
  s = v->text;
  if (!*s) return 0;
  for (; *s; s++) {
    uint64_t d;
    if (*s < '0' || *s > '9') return 0; /* '-', '.', 'e' */
    d = (uint64_t)(*s - '0');
    if (x > (limit - d) / 10) return 0;
    x = x * 10 + d;
  }
  *out = x;
  return 1;
}

/* ===================================================================== */
/* 2. The index: parse + validate.                                        */
/* ===================================================================== */

typedef struct {
  char *name;
  int dtype;
  int ndim;
  int64_t *shape;
  uint64_t numel;
  uint64_t begin, end; /* relative to the data section */
} or_entry;

typedef struct or_index {
  or_entry *e;
  uint64_t n;
  uint64_t header_len; /* N */
  uint64_t data_bytes;
  uint64_t nmeta;
  char **meta_keys;
  char **meta_vals;
} or_index;

static char *dupstr(const char *s) {
  size_t n = strlen(s);
  char *d = (char *)malloc(n + 1);
  if (d) memcpy(d, s, n + 1);
  return d;
}

void or_index_free(or_index *ix) {
  uint64_t i;
  if (!ix) return;
  for (i = 0; i < ix->n; i++) {
    free(ix->e[i].name);
    free(ix->e[i].shape);
  }
  for (i = 0; i < ix->nmeta; i++) {
    free(ix->meta_keys[i]);
    free(ix->meta_vals[i]);
  }
  free(ix->e);
  free(ix->meta_keys);
  free(ix->meta_vals);
  free(ix);
}

/* Index order: ascending begin, then end, then name (bytewise). */
static int entry_cmp(const void *a, const void *b) {
  const or_entry *x = (const or_entry *)a, *y = (const or_entry *)b;
  if (x->begin != y->begin) return x->begin < y->begin ? -1 : 1;
  if (x->end != y->end) return x->end < y->end ? -1 : 1;
  return strcmp(x->name, y->name);
}

/* Validates one tensor entry object `v` named `name`, filling `e`. */
static int check_entry(const char *name, const jval *v, uint64_t data_bytes, or_entry *e) {
  const jval *dt = NULL, *sh = NULL, *off = NULL;
  uint64_t numel = 1, nbytes, b, en;
  size_t i;
  int d;
  if (v->kind != J_OBJ) return OR_E_HEADER_JSON;
  for (i = 0; i < v->n; i++) {
    const jval **slot;
    if (strcmp(v->keys[i], "dtype") == 0) slot = &dt;
    else if (strcmp(v->keys[i], "shape") == 0) slot = &sh;
    else if (strcmp(v->keys[i], "data_offsets") == 0) slot = &off;
    else return OR_E_HEADER_JSON; /* unknown key */
    if (*slot) return OR_E_HEADER_JSON; /* repeated key */
    *slot = &v->items[i];
  }
  if (!dt || !sh || !off) return OR_E_HEADER_JSON;
  if (dt->kind != J_STR || sh->kind != J_ARR || off->kind != J_ARR || off->n != 2)
    return OR_E_HEADER_JSON;
  for (i = 0; i < sh->n; i++)
    if (sh->items[i].kind != J_NUM) return OR_E_HEADER_JSON;
  for (i = 0; i < 2; i++)
    if (off->items[i].kind != J_NUM) return OR_E_HEADER_JSON;
  /* dtype */
  for (d = 0; d < 15; d++)
    if (strcmp(dt->text, kNames[d]) == 0) break;
  if (d == 15) return OR_E_DTYPE;
  /* shape: non-negative integers, product (times itemsize) fits in 64 bits */
  e->shape = (int64_t *)malloc((sh->n ? sh->n : 1) * sizeof(int64_t));
  if (!e->shape) return OR_E_NOMEM;
  for (i = 0; i < sh->n; i++) {
    uint64_t dim;
    if (!jnum_to_u64(&sh->items[i], (uint64_t)INT64_MAX, &dim)) return OR_E_SHAPE;
    e->shape[i] = (int64_t)dim;
    if (dim != 0 && numel > UINT64_MAX / dim) return OR_E_SHAPE;
    numel *= dim;
  }
  if (numel > UINT64_MAX / (uint64_t)kSize[d]) return OR_E_SHAPE;
  nbytes = numel * (uint64_t)kSize[d];
  /* offsets */
  if (!jnum_to_u64(&off->items[0], UINT64_MAX, &b)) return OR_E_OFFSETS;
  if (!jnum_to_u64(&off->items[1], UINT64_MAX, &en)) return OR_E_OFFSETS;
  if (b > en || en > data_bytes || en - b != nbytes) return OR_E_OFFSETS;
  e->name = dupstr(name);
  if (!e->name) return OR_E_NOMEM;
  e->dtype = d;
  e->ndim = (int)sh->n;
  e->numel = numel;
  e->begin = b;
  e->end = en;
  return OR_OK;
}

static int check_metadata(const jval *v, or_index *ix) {
  size_t i, j;
  if (v->kind != J_OBJ) return OR_E_HEADER_JSON;
  for (i = 0; i < v->n; i++) {
    if (v->items[i].kind != J_STR) return OR_E_HEADER_JSON;
    for (j = 0; j < i; j++)
      if (strcmp(v->keys[i], v->keys[j]) == 0) return OR_E_HEADER_JSON;
  }
  ix->nmeta = v->n;
  ix->meta_keys = (char **)calloc(v->n ? v->n : 1, sizeof(char *));
  ix->meta_vals = (char **)calloc(v->n ? v->n : 1, sizeof(char *));
  if (!ix->meta_keys || !ix->meta_vals) return OR_E_NOMEM;
  for (i = 0; i < v->n; i++) {
    ix->meta_keys[i] = dupstr(v->keys[i]);
    ix->meta_vals[i] = dupstr(v->items[i].text);
  }
  return OR_OK;
}

/* Reads the 8-byte little-endian header length. */
static uint64_t read_u64le(const uint8_t *p) {
  uint64_t x = 0;
  int i;
  for (i = 7; i >= 0; i--) x = (x << 8) | p[i];
  return x;
}

typedef struct {
  const char *name;
  uint64_t pos;
} name_pos;

static int name_pos_cmp(const void *a, const void *b) {
  const name_pos *x = (const name_pos *)a, *y = (const name_pos *)b;
  int c = strcmp(x->name, y->name);
  if (c) return c;
  return x->pos < y->pos ? -1 : (x->pos > y->pos);
}

/* repeated[i] = 1 when member i's key already appeared at an earlier member. */
static char *mark_repeats(char **keys, uint64_t n) {
  char *rep = (char *)calloc(n ? n : 1, 1);
  name_pos *v = (name_pos *)malloc((n ? n : 1) * sizeof(name_pos));
  uint64_t i;
  if (!rep || !v) { free(rep); free(v); return NULL; }
  for (i = 0; i < n; i++) { v[i].name = keys[i]; v[i].pos = i; }
  qsort(v, n, sizeof(name_pos), name_pos_cmp);
  for (i = 1; i < n; i++)
    if (strcmp(v[i].name, v[i - 1].name) == 0) rep[v[i].pos] = 1;
  free(v);
  return rep;
}

/* Parses the first 8 + N bytes of a file (`len` of them given) whose data
   section is `data_bytes` long. */
int or_parse_header(const uint8_t *file, uint64_t len, uint64_t data_bytes, or_index **out) {
  uint64_t N, i, expect;
  jreader r;
  jval root;
  or_index *ix;
  char *repeated;
  int st = OR_OK;
  *out = NULL;
  if (len < 8) return OR_E_TRUNCATED;
  N = read_u64le(file);
  if (N > OR_MAX_HEADER) return OR_E_HEADER_TOO_LARGE;
  if (N > len - 8) return OR_E_TRUNCATED;
  r.p = file + 8;
  r.end = file + 8 + N;
  r.depth = 0;
  if (!jread_value(&r, &root)) { jfree(&root); return OR_E_HEADER_JSON; }
  jskip_ws(&r);
  if (r.p != r.end) { jfree(&root); return OR_E_HEADER_JSON; }
  if (root.kind != J_OBJ) { jfree(&root); return OR_E_HEADER_JSON; }
  ix = (or_index *)calloc(1, sizeof(or_index));
  if (!ix) { jfree(&root); return OR_E_NOMEM; }
  ix->header_len = N;
  ix->data_bytes = data_bytes;
  ix->e = (or_entry *)calloc(root.n ? root.n : 1, sizeof(or_entry));
  if (!ix->e) { jfree(&root); free(ix); return OR_E_NOMEM; }
  repeated = mark_repeats(root.keys, root.n);
  if (!repeated) { jfree(&root); or_index_free(ix); return OR_E_NOMEM; }
  /* Members in document order; the first failure wins.  A key seen before
     (a tensor name or a second "__metadata__") is a duplicate. */
  for (i = 0; i < root.n && st == OR_OK; i++) {
    const char *name = root.keys[i];
    if (repeated[i]) { st = OR_E_DUP_KEY; break; }
    if (strcmp(name, "__metadata__") == 0) {
      st = check_metadata(&root.items[i], ix);
      continue;
    }
    st = check_entry(name, &root.items[i], data_bytes, &ix->e[ix->n]);
    ix->n++; /* counted even on failure so that free() releases it */
  }
  free(repeated);
  jfree(&root);
  if (st != OR_OK) { or_index_free(ix); return st; }
  /* Contiguity: sorted by offsets, the ranges tile [0, data_bytes) exactly. */
  qsort(ix->e, ix->n, sizeof(or_entry), entry_cmp);
  expect = 0;
  for (i = 0; i < ix->n; i++) {
    if (ix->e[i].begin != expect) { or_index_free(ix); return OR_E_OFFSETS; }
    expect = ix->e[i].end;
  }
  if (expect != data_bytes) { or_index_free(ix); return OR_E_OFFSETS; }
  *out = ix;
  return OR_OK;
}

/* Parses a whole file image (header length, JSON header, data section). */
int or_parse(const uint8_t *file, uint64_t file_len, or_index **out) {
  uint64_t N;
  *out = NULL;
  if (file_len < 8) return OR_E_TRUNCATED;
  N = read_u64le(file);
  if (N > OR_MAX_HEADER) return OR_E_HEADER_TOO_LARGE;
  if (N > file_len - 8) return OR_E_TRUNCATED;
  return or_parse_header(file, 8 + N, file_len - 8 - N, out);
}

/* --- accessors (for ctypes) --- */
uint64_t or_count(const or_index *ix) { return ix->n; }
uint64_t or_header_len(const or_index *ix) { return ix->header_len; }
uint64_t or_data_bytes(const or_index *ix) { return ix->data_bytes; }
const char *or_name(const or_index *ix, uint64_t i) { return ix->e[i].name; }
int or_dtype(const or_index *ix, uint64_t i) { return ix->e[i].dtype; }
int or_ndim(const or_index *ix, uint64_t i) { return ix->e[i].ndim; }
int64_t or_dim(const or_index *ix, uint64_t i, int d) { return ix->e[i].shape[d]; }
uint64_t or_numel(const or_index *ix, uint64_t i) { return ix->e[i].numel; }
uint64_t or_begin(const or_index *ix, uint64_t i) { return ix->e[i].begin; }
uint64_t or_end(const or_index *ix, uint64_t i) { return ix->e[i].end; }
uint64_t or_meta_count(const or_index *ix) { return ix->nmeta; }
const char *or_meta_key(const or_index *ix, uint64_t i) { return ix->meta_keys[i]; }
const char *or_meta_val(const or_index *ix, uint64_t i) { return ix->meta_vals[i]; }

/* Linear search by name; -1 when absent. */
int64_t or_find(const or_index *ix, const char *name) {
  uint64_t i;
  for (i = 0; i < ix->n; i++)
    if (strcmp(ix->e[i].name, name) == 0) return (int64_t)i;
  return -1;
}

/* ===================================================================== */
/* 3. Views ("Strategy summary": PrefixView / FilterView / RenameView).   */
/*    A view is a new index holding copies of the selected entries under  */
/*    their new names, in the parent's order.                             */
/* ===================================================================== */

static or_index *view_alloc(const or_index *parent) {
  or_index *v = (or_index *)calloc(1, sizeof(or_index));
  if (!v) return NULL;
  v->e = (or_entry *)calloc(parent->n ? parent->n : 1, sizeof(or_entry));
  if (!v->e) { free(v); return NULL; }
  v->header_len = parent->header_len;
  v->data_bytes = parent->data_bytes;
  return v;
}

static int view_add(or_index *v, const or_entry *src, const char *newname) {
  or_entry *d = &v->e[v->n];
  *d = *src;
  d->name = dupstr(newname);
  d->shape = (int64_t *)malloc((src->ndim ? src->ndim : 1) * sizeof(int64_t));
  if (!d->name || !d->shape) return OR_E_NOMEM;
  memcpy(d->shape, src->shape, (size_t)src->ndim * sizeof(int64_t));
  v->n++;
  return OR_OK;
}

/* Prefix view: keeps names starting with `prefix` and strips it (reading of
   how BaseModel.load_model_weights consumes a prefix). */
int or_view_prefix(const or_index *parent, const char *prefix, or_index **out) {
  size_t k = strlen(prefix);
  uint64_t i;
  or_index *v = view_alloc(parent);
  if (!v) return OR_E_NOMEM;
  for (i = 0; i < parent->n; i++)
    if (strncmp(parent->e[i].name, prefix, k) == 0)
      if (view_add(v, &parent->e[i], parent->e[i].name + k) != OR_OK) { or_index_free(v); return OR_E_NOMEM; }
  *out = v;
  return OR_OK;
}

/* Filter view: keeps the listed names (each must exist), in parent order. */
int or_view_filter(const or_index *parent, const char *const *names, uint64_t n, or_index **out) {
  uint64_t i, j;
  or_index *v;
  for (j = 0; j < n; j++)
    if (or_find(parent, names[j]) < 0) return OR_E_NOT_FOUND;
  v = view_alloc(parent);
  if (!v) return OR_E_NOMEM;
  for (i = 0; i < parent->n; i++) {
    int keep = 0;
    for (j = 0; j < n && !keep; j++)
      if (strcmp(parent->e[i].name, names[j]) == 0) keep = 1;
    if (keep && view_add(v, &parent->e[i], parent->e[i].name) != OR_OK) { or_index_free(v); return OR_E_NOMEM; }
  }
  *out = v;
  return OR_OK;
}

/* Rename view: ordered (from-prefix -> to-prefix) rules, the first matching
   rule wins, unmatched names are kept (state_dict_prefix_replace).  Two
   entries that end up with the same name are an error. */
int or_view_rename(const or_index *parent, const char *const *from, const char *const *to, uint64_t n,
                   or_index **out) {
  uint64_t i, j;
  or_index *v = view_alloc(parent);
  if (!v) return OR_E_NOMEM;
  for (i = 0; i < parent->n; i++) {
    const char *nm = parent->e[i].name;
    char *buf = NULL;
    int st;
    for (j = 0; j < n; j++) {
      size_t k = strlen(from[j]);
      if (strncmp(nm, from[j], k) == 0) {
        size_t a = strlen(to[j]), b = strlen(nm + k);
        buf = (char *)malloc(a + b + 1);
        if (!buf) { or_index_free(v); return OR_E_NOMEM; }
        memcpy(buf, to[j], a);
        memcpy(buf + a, nm + k, b + 1);
        break;
      }
    }
    st = view_add(v, &parent->e[i], buf ? buf : nm);
    free(buf);
    if (st != OR_OK) { or_index_free(v); return st; }
  }
  for (i = 0; i < v->n; i++)
    for (j = 0; j < i; j++)
      if (strcmp(v->e[i].name, v->e[j].name) == 0) { or_index_free(v); return OR_E_DUP_KEY; }
  *out = v;
  return OR_OK;
}

/* Joined index over shard files ("Strategy summary (implemented)": one
   streaming mapping over a checkpoint split in shards).  Reading: shard k's
   data section sits in one arena at bases[k], the previous shard's end
   rounded up to a multiple of `align`; the joined index lists every part's
   entries in part order with offsets shifted by the part's base; a name in
   two parts is an error; metadata keeps a key's first occurrence. */
int or_concat(const or_index *const *parts, uint64_t n, uint64_t align, uint64_t *bases, or_index **out) {
  uint64_t k, i, j, total = 0, metas = 0, end = 0;
  or_index *v;
  if (n == 0 || align == 0 || (align & (align - 1)) != 0) return OR_E_INVAL;
  for (k = 0; k < n; k++) {
    total += parts[k]->n;
    metas += parts[k]->nmeta;
  }
  v = (or_index *)calloc(1, sizeof(or_index));
  if (!v) return OR_E_NOMEM;
  v->e = (or_entry *)calloc(total ? total : 1, sizeof(or_entry));
  v->meta_keys = (char **)calloc(metas ? metas : 1, sizeof(char *));
  v->meta_vals = (char **)calloc(metas ? metas : 1, sizeof(char *));
  if (!v->e || !v->meta_keys || !v->meta_vals) { or_index_free(v); return OR_E_NOMEM; }
  for (k = 0; k < n; k++) {
    const or_index *p = parts[k];
    uint64_t base = end;
    while (base % align != 0) base++;
    bases[k] = base;
    end = base + p->data_bytes;
    for (i = 0; i < p->n; i++) {
      if (view_add(v, &p->e[i], p->e[i].name) != OR_OK) { or_index_free(v); return OR_E_NOMEM; }
      v->e[v->n - 1].begin += base;
      v->e[v->n - 1].end += base;
    }
    for (i = 0; i < p->nmeta; i++) {
      int seen = 0;
      for (j = 0; j < v->nmeta; j++)
        if (strcmp(v->meta_keys[j], p->meta_keys[i]) == 0) seen = 1;
      if (seen) continue;
      v->meta_keys[v->nmeta] = dupstr(p->meta_keys[i]);
      v->meta_vals[v->nmeta] = dupstr(p->meta_vals[i]);
      v->nmeta++;
      if (!v->meta_keys[v->nmeta - 1] || !v->meta_vals[v->nmeta - 1]) { or_index_free(v); return OR_E_NOMEM; }
    }
  }
  v->data_bytes = end;
  v->header_len = 0;
  for (i = 0; i < v->n; i++)
    for (j = 0; j < i; j++)
      if (strcmp(v->e[i].name, v->e[j].name) == 0) { or_index_free(v); return OR_E_DUP_KEY; }
  *out = v;
  return OR_OK;
}

/* ===================================================================== */
/* 4. Float formats: exact decode, round-to-nearest-even encode.          */
/* ===================================================================== */

static int is_float(int dt) {
  return dt == OR_F16 || dt == OR_BF16 || dt == OR_F32 || dt == OR_F64 || dt == OR_F8_E4M3 ||
         dt == OR_F8_E5M2;
}
static int is_fp8(int dt) { return dt == OR_F8_E4M3 || dt == OR_F8_E5M2; }

/* IEEE-style interchange format with `eb` exponent bits, `mb` fraction bits:
   all-ones exponent is infinity (zero fraction) or NaN. */
static double decode_ieee(uint64_t bits, int eb, int mb, int *nan) {
  int bias = (1 << (eb - 1)) - 1;
  uint64_t s = (bits >> (eb + mb)) & 1;
  uint64_t e = (bits >> mb) & ((1ull << eb) - 1);
  uint64_t m = bits & ((1ull << mb) - 1);
  double mag;
  *nan = 0;
  if (e == (1ull << eb) - 1) {
    if (m != 0) { *nan = 1; return NAN; }
    mag = INFINITY;
  } else if (e == 0) {
    mag = ldexp((double)m, 1 - bias - mb); /* subnormal: m * 2^(1-bias-mb) */
  } else {
    mag = ldexp((double)((1ull << mb) | m), (int)e - bias - mb);
  }
  return s ? -mag : mag;
}

/* OCP E4M3 ("fn"): bias 7, no infinities, S.1111.111 is the only NaN. */
static double decode_e4m3(uint64_t bits, int *nan) {
  uint64_t s = (bits >> 7) & 1, e = (bits >> 3) & 15, m = bits & 7;
  double mag;
  *nan = 0;
  if (e == 15 && m == 7) { *nan = 1; return NAN; }
  if (e == 0) mag = ldexp((double)m, 1 - 7 - 3);
  else mag = ldexp((double)(8 | m), (int)e - 7 - 3);
  return s ? -mag : mag;
}

/* Exact value of one element of a float dtype. */
static double decode_value(int dt, uint64_t bits, int *nan) {
  switch (dt) {
    case OR_F16: return decode_ieee(bits, 5, 10, nan);
    case OR_BF16: return decode_ieee(bits, 8, 7, nan);
    case OR_F32: return decode_ieee(bits, 8, 23, nan);
    case OR_F8_E5M2: return decode_ieee(bits, 5, 2, nan);
    case OR_F8_E4M3: return decode_e4m3(bits, nan);
    default: *nan = 1; return NAN;
  }
}

/* Rounds the exact value v to the IEEE-style format (eb, mb): nearest
   representable value, ties to the even significand, gradual underflow,
   overflow to infinity.  NaN becomes the positive quiet NaN. */
static uint64_t encode_rne(double v, int nan, int eb, int mb) {
  int bias = (1 << (eb - 1)) - 1;
  int emin = 1 - bias, emax = bias;
  uint64_t sign = 0, expall = (1ull << eb) - 1, m;
  double a, q, n, fl, frac;
  int E;
  if (nan || v != v) return (expall << mb) | (1ull << (mb - 1));
  if (signbit(v)) { sign = 1ull << (eb + mb); a = -v; } else a = v;
  if (isinf(a)) return sign | (expall << mb);
  if (a == 0.0) return sign;
  (void)frexp(a, &E);
  E -= 1;                        /* a in [2^E, 2^(E+1)) */
  if (E < emin) E = emin;        /* subnormal range shares emin's quantum */
  q = ldexp(1.0, E - mb);        /* spacing of representable values */
  n = a / q;                     /* exact: q is a power of two */
  fl = floor(n);
  frac = n - fl;
  m = (uint64_t)fl;
  if (frac > 0.5 || (frac == 0.5 && (m & 1))) m += 1;
  if (m == (1ull << (mb + 1))) { m >>= 1; E += 1; } /* carried into the next binade */
  if (E > emax) return sign | (expall << mb);        /* overflow */
  if (m < (1ull << mb)) return sign | m;             /* subnormal or zero */
  return sign | ((uint64_t)(E + bias) << mb) | (m - (1ull << mb));
}

static uint64_t encode_to(int dt, double v, int nan) {
  switch (dt) {
    case OR_BF16: return encode_rne(v, nan, 8, 7);
    case OR_F16: return encode_rne(v, nan, 5, 10);
    default: return encode_rne(v, nan, 8, 23); /* OR_F32 */
  }
}

static uint64_t load_le(const uint8_t *p, int n) {
  uint64_t x = 0;
  int i;
  for (i = n - 1; i >= 0; i--) x = (x << 8) | p[i];
  return x;
}
static void store_le(uint8_t *p, uint64_t x, int n) {
  int i;
  for (i = 0; i < n; i++) { p[i] = (uint8_t)(x & 0xFF); x >>= 8; }
}

/* Output dtype of a tensor of dtype `src` materialized with target `req`:
   integers and bool keep their dtype ("ints/bool copied raw"), KEEP keeps
   every dtype, and float sources take the requested float dtype.  Returns -1
   for an unsupported request. */
int or_out_dtype(int src, int req) {
  if (src < 0 || src >= 15) return -1;
  if (req == OR_KEEP || !is_float(src)) return src;
  if (req != OR_BF16 && req != OR_F16 && req != OR_F32) return -1;
  if (src == OR_F64) return req == OR_F64 ? src : -1;
  return req;
}

/* Converts n elements.  With `scaled` set (fp8 sources only) every element is
   decoded, converted to binary32 (exact), multiplied by `scale` with a single
   binary32 multiply, then rounded to the output dtype.  A source equal to the
   output dtype without a scale is a byte copy. */
int or_convert(int src, int out, const uint8_t *in, uint64_t n, int scaled, float scale, uint8_t *dst) {
  int si, so;
  uint64_t i;
  if (src < 0 || src >= 15 || out < 0 || out >= 15) return OR_E_INVAL;
  si = kSize[src];
  so = kSize[out];
  if (scaled && !is_fp8(src)) return OR_E_INVAL;
  if (src == out && !scaled) {
    memcpy(dst, in, (size_t)(n * (uint64_t)si));
    return OR_OK;
  }
  if (!is_float(src) || src == OR_F64 || (out != OR_BF16 && out != OR_F16 && out != OR_F32))
    return OR_E_UNSUPPORTED_CAST;
  for (i = 0; i < n; i++) {
    int nan;
    double x = decode_value(src, load_le(in + i * (uint64_t)si, si), &nan);
    uint64_t bits;
    if (is_fp8(src)) {
      float xf = (float)x;           /* exact: every fp8 value is a binary32 value */
      float s = scaled ? scale : 1.0f;
      float p = xf * s;              /* the one binary32 multiply */
      bits = encode_to(out, (double)p, nan || p != p);
    } else {
      bits = encode_to(out, x, nan);
    }
    store_le(dst + i * (uint64_t)so, bits, so);
  }
  return OR_OK;
}

/* ===================================================================== */
/* 5. Selection and plan: which outputs, in which order, with which scale. */
/* ===================================================================== */

/* Block-scaled weight formats (an output of one of them reads a second
   tensor of scales): */
enum { OR_Q_NONE = 0, OR_Q_BLOCK_FP8 = 2, OR_Q_NVFP4 = 3 };

typedef struct {
  char *name;       /* output name (the index/view name) */
  uint64_t entry;   /* index entry */
  int out_dtype;
  int64_t scale;    /* index entry of the f32 scale, or -1 */
  int sdim;         /* sliced dimension, or -1 */
  int64_t start, stop;
  uint64_t numel;   /* elements of the output (after slicing) */
  int qkind;        /* OR_Q_* */
  int64_t qscale;   /* block scales tensor, or -1 */
  int64_t qscale2;  /* NVFP4 global scale tensor, or -1 */
  uint64_t br, bc;  /* block rows, block columns (elements) */
  uint64_t rows, cols;  /* the output as a matrix */
} or_output;

/* Products of the dimensions before and after `dim`. */
static void outer_inner(const or_entry *e, int dim, uint64_t *outer, uint64_t *inner) {
  int d;
  *outer = 1;
  *inner = 1;
  for (d = 0; d < dim; d++) *outer *= (uint64_t)e->shape[d];
  for (d = dim + 1; d < e->ndim; d++) *inner *= (uint64_t)e->shape[d];
}

typedef struct or_plan {
  or_output *o;
  uint64_t n;
} or_plan;

void or_plan_free(or_plan *p) {
  uint64_t i;
  if (!p) return;
  for (i = 0; i < p->n; i++) free(p->o[i].name);
  free(p->o);
  free(p);
}

static int ends_with(const char *s, const char *suf) {
  size_t a = strlen(s), b = strlen(suf);
  return a >= b && strcmp(s + a - b, suf) == 0;
}

/* names == NULL selects every entry in index order.  slices (when not NULL,
   with names) holds three numbers per name: dim, start, stop; the output is
   then the tensor's [start, stop) range along dim (dim < 0: the whole
   tensor), each [0, ndim), 0 <= start <= stop <= shape[dim].  scale_names
   (when not NULL) gives each selected name its scale tensor (NULL for none).  Otherwise,
   when both suffixes are given, an fp8 tensor "<stem><from>" is paired with
   "<stem><to>" if that tensor exists.  A scale must be a one-element F32
   tensor and may only scale an fp8 tensor.  Tensors used as scales are
   consumed: they are not outputs.  Optionally keeps only part `part` of
   `nparts` (balanced by output bytes, contiguous in output order). */
static int is_pow2(uint64_t v) { return v != 0 && (v & (v - 1)) == 0; }

/* Checks the block-scaled format of selected name i and fills its output
   fields (reading: the formats are only named on the pages).
     OR_Q_BLOCK_FP8: an fp8 [M, N] weight and an F32 [ceil(M/br), ceil(N/bc)]
       scale tensor; element (i, j) is multiplied by scale (i/br, j/bc).
       Block sizes are powers of two, bc >= 16 (0: 128).
     OR_Q_NVFP4: a U8 [M, K] weight holding M x 2K e2m1 values (element 2c in
       the low nibble of byte c, 2c+1 in the high nibble), an F8_E4M3
       [M, ceil(2K/16)] tensor of block scales (16 elements along a row) and a
       one-element F32 global scale. */
static int check_quant(const or_index *ix, const or_entry *e, int kind, const char *qs, const char *qs2,
                       uint64_t br, uint64_t bc, or_output *o, char *consumed) {
  int64_t si, si2 = -1;
  const or_entry *sc;
  if (kind != OR_Q_BLOCK_FP8 && kind != OR_Q_NVFP4) return OR_E_INVAL;
  if (!qs) return OR_E_INVAL;
  si = or_find(ix, qs);
  if (si < 0) return OR_E_NOT_FOUND;
  sc = &ix->e[si];
  if (e->ndim != 2) return OR_E_INVAL;
  o->rows = (uint64_t)e->shape[0];
  if (kind == OR_Q_BLOCK_FP8) {
    if (br == 0) br = 128;
    if (bc == 0) bc = 128;
    if (!is_fp8(e->dtype) || !is_pow2(br) || !is_pow2(bc) || bc < 16) return OR_E_INVAL;
    o->cols = (uint64_t)e->shape[1];
    if (sc->dtype != OR_F32 || sc->ndim != 2 || (uint64_t)sc->shape[0] != (o->rows + br - 1) / br ||
        (uint64_t)sc->shape[1] != (o->cols + bc - 1) / bc)
      return OR_E_INVAL;
  } else {
    if (!((br == 0 && bc == 0) || (br == 1 && bc == 16))) return OR_E_INVAL;
    br = 1;
    bc = 16;
    if (e->dtype != OR_U8 || !qs2) return OR_E_INVAL;
    si2 = or_find(ix, qs2);
    if (si2 < 0) return OR_E_NOT_FOUND;
    o->cols = 2 * (uint64_t)e->shape[1];
    if (sc->dtype != OR_F8_E4M3 || sc->ndim != 2 || (uint64_t)sc->shape[0] != o->rows ||
        (uint64_t)sc->shape[1] != (o->cols + 15) / 16)
      return OR_E_INVAL;
    if (ix->e[si2].dtype != OR_F32 || ix->e[si2].numel != 1) return OR_E_INVAL;
    consumed[si2] = 1;
  }
  consumed[si] = 1;
  o->qkind = kind;
  o->qscale = si;
  o->qscale2 = si2;
  o->br = br;
  o->bc = bc;
  o->numel = o->rows * o->cols;
  return OR_OK;
}

int or_select_q(const or_index *ix, const char *const *names, uint64_t n_names,
                const char *const *scale_names, const char *from, const char *to, int req,
                uint64_t part, uint64_t nparts, const int64_t *slices, const int *qkind,
                const char *const *qscale, const char *const *qscale2, const int64_t *qblock, or_plan **out) {
  uint64_t n = names ? n_names : ix->n, i, j, k;
  int64_t *ent = NULL, *sc = NULL;
  char *consumed = NULL;
  or_output *qo = NULL;
  or_plan *p = NULL;
  int st = OR_OK;
  *out = NULL;
  if (nparts == 0 || part >= nparts) return OR_E_INVAL;
  if (req != OR_BF16 && req != OR_F16 && req != OR_F32 && req != OR_KEEP) return OR_E_UNSUPPORTED_CAST;
  ent = (int64_t *)malloc((n ? n : 1) * sizeof(int64_t));
  sc = (int64_t *)malloc((n ? n : 1) * sizeof(int64_t));
  consumed = (char *)calloc(ix->n ? ix->n : 1, 1);
  if (!ent || !sc || !consumed) { st = OR_E_NOMEM; goto done; }
  for (i = 0; i < n; i++) {
    ent[i] = names ? or_find(ix, names[i]) : (int64_t)i;
    if (ent[i] < 0) { st = OR_E_NOT_FOUND; goto done; }
    for (j = 0; j < i; j++)
      if (ent[j] == ent[i]) { st = OR_E_DUP_KEY; goto done; }
    sc[i] = -1;
  }
  if (slices && !names) { st = OR_E_INVAL; goto done; }
  for (i = 0; slices && i < n; i++) {
    const or_entry *e = &ix->e[ent[i]];
    int64_t dim = slices[3 * i], a = slices[3 * i + 1], b = slices[3 * i + 2];
    if (dim < 0) continue;
    if (dim >= e->ndim || a < 0 || a > b || b > e->shape[dim]) { st = OR_E_INVAL; goto done; }
  }
  /* Block-scaled formats: explicit per name; not sliced, no per-tensor scale,
     and only to a float dtype. */
  if (qkind && !names) { st = OR_E_INVAL; goto done; }
  qo = (or_output *)calloc(n ? n : 1, sizeof(or_output));
  if (!qo) { st = OR_E_NOMEM; goto done; }
  for (i = 0; qkind && i < n; i++) {
    if (qkind[i] == OR_Q_NONE) continue;
    if ((slices && slices[3 * i] >= 0) || (scale_names && scale_names[i])) { st = OR_E_INVAL; goto done; }
    if (req == OR_KEEP) { st = OR_E_UNSUPPORTED_CAST; goto done; }
    st = check_quant(ix, &ix->e[ent[i]], qkind[i], qscale ? qscale[i] : NULL, qscale2 ? qscale2[i] : NULL,
                     qblock ? (uint64_t)qblock[2 * i] : 0, qblock ? (uint64_t)qblock[2 * i + 1] : 0, &qo[i],
                     consumed);
    if (st != OR_OK) goto done;
  }
  for (i = 0; i < n; i++) {
    const or_entry *e = &ix->e[ent[i]];
    if (qo[i].qkind != OR_Q_NONE) continue;
    if (scale_names) {
      if (scale_names[i]) {
        sc[i] = or_find(ix, scale_names[i]);
        if (sc[i] < 0) { st = OR_E_NOT_FOUND; goto done; }
      }
    } else if (from && to && is_fp8(e->dtype) && ends_with(e->name, from)) {
      size_t stem = strlen(e->name) - strlen(from), tl = strlen(to);
      char *cand = (char *)malloc(stem + tl + 1);
      if (!cand) { st = OR_E_NOMEM; goto done; }
      memcpy(cand, e->name, stem);
      memcpy(cand + stem, to, tl + 1);
      sc[i] = or_find(ix, cand);
      free(cand);
    }
    if (sc[i] >= 0) {
      const or_entry *s = &ix->e[sc[i]];
      if (!is_fp8(e->dtype) || s->dtype != OR_F32 || s->numel != 1) { st = OR_E_INVAL; goto done; }
      if (req == OR_KEEP) { st = OR_E_UNSUPPORTED_CAST; goto done; }
      consumed[sc[i]] = 1;
    }
  }
  p = (or_plan *)calloc(1, sizeof(or_plan));
  if (!p) { st = OR_E_NOMEM; goto done; }
  p->o = (or_output *)calloc(n ? n : 1, sizeof(or_output));
  if (!p->o) { st = OR_E_NOMEM; goto done; }
  for (i = 0; i < n; i++) {
    const or_entry *e = &ix->e[ent[i]];
    int od;
    if (consumed[ent[i]]) continue;
    od = or_out_dtype(e->dtype, req);
    if (od < 0) { st = OR_E_UNSUPPORTED_CAST; goto done; }
    p->o[p->n] = qo[i];
    p->o[p->n].name = dupstr(e->name);
    p->o[p->n].entry = (uint64_t)ent[i];
    p->o[p->n].out_dtype = qo[i].qkind != OR_Q_NONE ? req : od;
    p->o[p->n].scale = sc[i];
    p->o[p->n].sdim = -1;
    if (qo[i].qkind == OR_Q_NONE) {
      p->o[p->n].numel = e->numel;
      p->o[p->n].qscale = p->o[p->n].qscale2 = -1;
    }
    if (slices && slices[3 * i] >= 0) {
      uint64_t outer, inner;
      int dim = (int)slices[3 * i];
      outer_inner(e, dim, &outer, &inner);
      p->o[p->n].sdim = dim;
      p->o[p->n].start = slices[3 * i + 1];
      p->o[p->n].stop = slices[3 * i + 2];
      p->o[p->n].numel = outer * (uint64_t)(slices[3 * i + 2] - slices[3 * i + 1]) * inner;
    }
    p->n++;
  }
  if (nparts > 1) {
    /* Output i (bytes b_i, c_i bytes before it, total T) goes to part
       floor(nparts * (c_i + b_i / 2) / T), computed as
       floor(nparts * (2 c_i + b_i) / (2 T)); with T == 0 all go to part 0. */
    unsigned __int128 T = 0, c = 0;
    for (i = 0; i < p->n; i++) T += (unsigned __int128)p->o[i].numel * kSize[p->o[i].out_dtype];
    for (i = 0, k = 0; i < p->n; i++) {
      unsigned __int128 b = (unsigned __int128)p->o[i].numel * kSize[p->o[i].out_dtype];
      uint64_t owner = 0;
      if (T > 0) {
        unsigned __int128 q = ((2 * c + b) * nparts) / (2 * T);
        owner = (uint64_t)(q >= nparts ? nparts - 1 : q);
      }
      c += b;
      if (owner == part) p->o[k++] = p->o[i];
      else free(p->o[i].name);
    }
    p->n = k;
  }
  *out = p;
  p = NULL;
done:
  free(ent);
  free(sc);
  free(consumed);
  free(qo);
  or_plan_free(p);
  return st;
}

int or_select(const or_index *ix, const char *const *names, uint64_t n_names,
              const char *const *scale_names, const char *from, const char *to, int req,
              uint64_t part, uint64_t nparts, const int64_t *slices, or_plan **out) {
  return or_select_q(ix, names, n_names, scale_names, from, to, req, part, nparts, slices, NULL, NULL, NULL, NULL,
                     out);
}

int or_plan_quant(const or_plan *p, uint64_t i) { return p->o[i].qkind; }
int64_t or_plan_qscale(const or_plan *p, uint64_t i) { return p->o[i].qscale; }
int64_t or_plan_qscale2(const or_plan *p, uint64_t i) { return p->o[i].qscale2; }

uint64_t or_plan_count(const or_plan *p) { return p->n; }
const char *or_plan_name(const or_plan *p, uint64_t i) { return p->o[i].name; }
uint64_t or_plan_entry(const or_plan *p, uint64_t i) { return p->o[i].entry; }
int or_plan_dtype(const or_plan *p, uint64_t i) { return p->o[i].out_dtype; }
int64_t or_plan_scale(const or_plan *p, uint64_t i) { return p->o[i].scale; }

/* Elements and shape of output i (the sliced shape when sliced). */
uint64_t or_plan_numel(const or_plan *p, uint64_t i) { return p->o[i].numel; }
int or_plan_ndim(const or_index *ix, const or_plan *p, uint64_t i) { return ix->e[p->o[i].entry].ndim; }
int64_t or_plan_dim(const or_index *ix, const or_plan *p, uint64_t i, int d) {
  const or_output *o = &p->o[i];
  if (o->qkind != OR_Q_NONE) return d == 0 ? (int64_t)o->rows : (int64_t)o->cols;
  if (d == o->sdim) return o->stop - o->start;
  return ix->e[o->entry].shape[d];
}

/* Bytes of output i. */
uint64_t or_plan_bytes(const or_index *ix, const or_plan *p, uint64_t i) {
  (void)ix;
  return p->o[i].numel * (uint64_t)kSize[p->o[i].out_dtype];
}

/* Converts output elements [first, first + count) of output o (source
   element index of output element e: the row e / run of the slice, then the
   column e % run, run = (stop - start) * inner elements per row). */
/* OCP MX E2M1 (FP4): sign, 2 exponent bits (bias 1), 1 mantissa bit; no
   infinities or NaN. */
static double decode_e2m1(unsigned nib) {
  unsigned sgn = (nib >> 3) & 1, ex = (nib >> 1) & 3, m = nib & 1;
  double v = ex == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, (int)ex - 1);
  return sgn ? -v : v;
}

static float load_f32(const uint8_t *p) {
  uint32_t u = (uint32_t)load_le(p, 4);
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Output element (i, j) of a block-scaled output: the weight value times its
   block's scale, each product one binary32 multiply (NVFP4: the block scale
   times the global scale first, then the value times that). */
static void convert_quant(const or_index *ix, const or_output *o, const uint8_t *data, uint64_t first,
                          uint64_t count, uint8_t *dst) {
  const or_entry *e = &ix->e[o->entry], *sc = &ix->e[o->qscale];
  const int so = kSize[o->out_dtype];
  const uint64_t scols = (uint64_t)sc->shape[1];
  uint64_t k;
  for (k = 0; k < count; k++) {
    const uint64_t oe = first + k, i = oe / o->cols, j = oe % o->cols;
    const uint64_t blk = (i / o->br) * scols + j / o->bc;
    int nan = 0;
    float v, s, x;
    if (o->qkind == OR_Q_BLOCK_FP8) {
      v = (float)decode_value(e->dtype, data[e->begin + oe], &nan);
      s = load_f32(data + sc->begin + 4 * blk);
    } else {
      const uint8_t byte = data[e->begin + i * (o->cols / 2) + j / 2];
      int snan = 0;
      const float sb = (float)decode_e4m3(data[sc->begin + blk], &snan);
      const float g = load_f32(data + ix->e[o->qscale2].begin);
      v = (float)decode_e2m1((j & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15));
      s = snan ? NAN : sb * g;
    }
    x = v * s;
    store_le(dst + k * (uint64_t)so, encode_to(o->out_dtype, (double)x, nan || x != x), so);
  }
}

static int convert_window(const or_index *ix, const or_output *o, const uint8_t *data, uint64_t first,
                          uint64_t count, uint8_t *dst) {
  const or_entry *e = &ix->e[o->entry];
  const int si = kSize[e->dtype], so = kSize[o->out_dtype];
  float scale = 1.0f;
  uint64_t done = 0;
  if (o->qkind != OR_Q_NONE) {
    convert_quant(ix, o, data, first, count, dst);
    return OR_OK;
  }
  if (o->scale >= 0) {
    const or_entry *s = &ix->e[o->scale];
    uint32_t u = (uint32_t)load_le(data + s->begin, 4);
    memcpy(&scale, &u, 4);
  }
  if (o->sdim < 0)
    return or_convert(e->dtype, o->out_dtype, data + e->begin + first * (uint64_t)si, count, o->scale >= 0, scale,
                      dst);
  {
    uint64_t outer, inner, run, D = (uint64_t)e->shape[o->sdim];
    outer_inner(e, o->sdim, &outer, &inner);
    run = (uint64_t)(o->stop - o->start) * inner;
    while (done < count) {
      uint64_t oe = first + done, row = oe / run, col = oe % run;
      uint64_t k = run - col < count - done ? run - col : count - done;
      uint64_t src_elem = (row * D + (uint64_t)o->start) * inner + col;
      int st = or_convert(e->dtype, o->out_dtype, data + e->begin + src_elem * si, k, o->scale >= 0, scale,
                          dst + done * so);
      if (st != OR_OK) return st;
      done += k;
    }
  }
  return OR_OK;
}

/* Materializes output i from the data section `data` (data_bytes long) into
   dst (or_plan_bytes(i) bytes). */
int or_materialize(const or_index *ix, const or_plan *p, uint64_t i, const uint8_t *data,
                   uint64_t data_bytes, uint8_t *dst) {
  const or_output *o = &p->o[i];
  if (ix->e[o->entry].end > data_bytes) return OR_E_OFFSETS;
  return convert_window(ix, o, data, 0, o->numel, dst);
}

/* Materializes a window [first, first + count) of output i's elements. */
int or_materialize_range(const or_index *ix, const or_plan *p, uint64_t i, const uint8_t *data,
                         uint64_t first, uint64_t count, uint8_t *dst) {
  const or_output *o = &p->o[i];
  if (first > o->numel || count > o->numel - first) return OR_E_INVAL;
  return convert_window(ix, o, data, first, count, dst);
}
