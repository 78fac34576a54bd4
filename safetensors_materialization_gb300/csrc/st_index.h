// st_index.h -- parsed header and index/view data shared by the host files.
#pragma once

#include <cstdint>
#include <deque>
#include <memory>
#include <string>
#include <string_view>
#include <unordered_map>
#include <utility>
#include <vector>

#include "stmat.h"

namespace stmat {

struct Tensor {
  std::string name;
  int dtype;
  std::vector<int64_t> shape;
  uint64_t numel;
  uint64_t begin, end;  // [begin, end) in the data section
};

// One parsed header: tensors in index order (begin, end, name).
struct Core {
  uint64_t header_len = 0;
  uint64_t data_bytes = 0;
  std::vector<Tensor> tensors;
  std::vector<std::pair<std::string, std::string>> meta;
};

// An index or a view: a selection of the core's tensors under names.
struct IndexData {
  std::shared_ptr<const Core> core;
  std::shared_ptr<const IndexData> parent;  // keeps the parent's name storage alive
  std::vector<uint32_t> ent;                // core tensor per position
  std::vector<const char *> names;          // name per position
  std::deque<std::string> owned;            // storage for renamed names
  std::unordered_map<std::string_view, uint32_t> pos;
};

size_t dtype_size(int dtype);
// A root index over `core` (positions = core order), and the name lookup of
// an index or view (ST_E_DUP_KEY on a repeated name).
std::shared_ptr<IndexData> make_root(std::shared_ptr<const Core> core);
st_status finish_view(IndexData *d);
const IndexData *index_data(const st_index *ix);
std::shared_ptr<const IndexData> index_ref(const st_index *ix);

}  // namespace stmat
