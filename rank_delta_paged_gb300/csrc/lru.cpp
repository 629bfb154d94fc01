// Recency index of resident adapters and its host-only C ABI.
//
// S-LoRA: Serving Thousands of Concurrent LoRA Adapters (explainer), "The mechanism":
// adapters that the running batches do not use can leave GPU memory and stay in host
// memory; "What to notice when reading": adapters and KV blocks compete for one pool.
// The pages do not name the policy that picks which adapters leave; this index takes the
// least recently used adapter that no running batch holds (pinned ones never leave).
// The pool uses it for slora_adapters_acquire and slora_pages_alloc_evict.  Needs no GPU.
#include <new>

#include "host_common.h"
#include "slora.h"

namespace slora {

int32_t LruIndex::pins(int32_t id) const
{
    auto it = ents.find(id);
    return it == ents.end() ? 0 : it->second.pins;
}

void LruIndex::insert(int32_t id)
{
    if (present(id))
        return;
    Ent e;
    e.last = ++clock;
    ents[id] = e;
    unpinned.insert({e.last, id});
}

void LruIndex::remove(int32_t id)
{
    auto it = ents.find(id);
    if (it == ents.end())
        return;
    if (it->second.pins == 0)
        unpinned.erase({it->second.last, id});
    ents.erase(it);
}

void LruIndex::touch(int32_t id)
{
    auto it = ents.find(id);
    if (it == ents.end())
        return;
    Ent &e = it->second;
    if (e.pins == 0)
        unpinned.erase({e.last, id});
    e.last = ++clock;
    if (e.pins == 0)
        unpinned.insert({e.last, id});
}

void LruIndex::pin(int32_t id)
{
    auto it = ents.find(id);
    if (it == ents.end())
        return;
    Ent &e = it->second;
    if (e.pins++ == 0)
        unpinned.erase({e.last, id});
}

bool LruIndex::unpin(int32_t id)
{
    auto it = ents.find(id);
    if (it == ents.end() || it->second.pins == 0)
        return false;
    Ent &e = it->second;
    if (--e.pins == 0)
        unpinned.insert({e.last, id});
    return true;
}

}  // namespace slora

using namespace slora;

struct slora_lru {
    LruIndex idx;
};

extern "C" {

slora_status slora_lru_create(slora_lru_t *out)
{
    if (!out)
        return fail(SLORA_ERR_INVALID_ARG, "lru_create: null out");
    *out = new (std::nothrow) slora_lru();
    return *out ? SLORA_OK : fail(SLORA_ERR_HOST_ALLOC, "lru_create");
}

slora_status slora_lru_destroy(slora_lru_t l)
{
    delete l;
    return SLORA_OK;
}

slora_status slora_lru_insert(slora_lru_t l, int32_t id)
{
    if (!l || id < 0)
        return fail(SLORA_ERR_INVALID_ARG, "lru_insert: id=%d", id);
    l->idx.insert(id);
    return SLORA_OK;
}

slora_status slora_lru_remove(slora_lru_t l, int32_t id)
{
    if (!l || !l->idx.present(id))
        return fail(SLORA_ERR_INVALID_ARG, "lru_remove: id=%d not present", id);
    if (l->idx.pins(id) > 0)
        return fail(SLORA_ERR_INVALID_ARG, "lru_remove: id=%d is pinned", id);
    l->idx.remove(id);
    return SLORA_OK;
}

slora_status slora_lru_touch(slora_lru_t l, int32_t id)
{
    if (!l || !l->idx.present(id))
        return fail(SLORA_ERR_INVALID_ARG, "lru_touch: id=%d not present", id);
    l->idx.touch(id);
    return SLORA_OK;
}

slora_status slora_lru_pin(slora_lru_t l, int32_t id)
{
    if (!l || !l->idx.present(id))
        return fail(SLORA_ERR_INVALID_ARG, "lru_pin: id=%d not present", id);
    l->idx.pin(id);
    return SLORA_OK;
}

slora_status slora_lru_unpin(slora_lru_t l, int32_t id)
{
    if (!l || !l->idx.unpin(id))
        return fail(SLORA_ERR_INVALID_ARG, "lru_unpin: id=%d not pinned", id);
    return SLORA_OK;
}

slora_status slora_lru_victims(slora_lru_t l, int32_t n_exclude, const int32_t *exclude, int32_t max_out,
                               int32_t *out_ids, int32_t *out_n)
{
    if (!l || n_exclude < 0 || (n_exclude > 0 && !exclude) || max_out < 0 || (max_out > 0 && !out_ids) || !out_n)
        return fail(SLORA_ERR_INVALID_ARG, "lru_victims");
    std::unordered_set<int32_t> ex(exclude, exclude + n_exclude);
    std::vector<int32_t> v;
    l->idx.victims(ex, [&](const std::vector<int32_t> &cur) { return (int32_t)cur.size() >= max_out; }, &v);
    for (size_t i = 0; i < v.size(); ++i)
        out_ids[i] = v[i];
    *out_n = (int32_t)v.size();
    return SLORA_OK;
}

}  // extern "C"
