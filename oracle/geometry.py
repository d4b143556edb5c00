"""KV-cache byte counts -- TEST INFRASTRUCTURE ONLY.

Source: "Tornar a inferência barata: KV cache, batching e quantização"
(neuralialabs.com), KV-cache memory paragraph: per context token, every
layer stores one key and one value vector per KV head, so a token costs
2 * layers * kv_heads * head_dim * bytes_per_element.  The same page checks it
against the allocator (3,624,960 bytes for 295 tokens of a 24-layer, 2-KV-head,
d = 64 fp16 model) and notes that the cache depends only on the total number
of resident tokens.
"""


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return 2 * layers * kv_heads * head_dim * elem_bytes


def kv_cache_bytes(tokens: int, layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return tokens * kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes)


def paged_pool_bytes(num_blocks: int, block_size: int, layers: int, kv_heads: int, head_dim: int,
                     elem_bytes: int) -> int:
    """K and V pools of num_blocks pages of block_size tokens, all layers."""
    return kv_cache_bytes(num_blocks * block_size, layers, kv_heads, head_dim, elem_bytes)
