"""Block-count, fragmentation and sharing arithmetic -- TEST INFRASTRUCTURE ONLY.

Plain restatements of the arithmetic the pages work through by hand:

* blocks for a sequence of T tokens: ceil(T / B); reserved slots B * ceil(T / B);
  waste below B slots per sequence ("PagedAttention: Virtual Memory for the KV
  Cache", "Where contiguous allocation wastes space" and "A block table
  preserves token order");
* paged versus contiguous-reservation fragmentation ("KV Cache Optimization and
  Management", "Worked Example 1" and active-recall answers A2, A3);
* blocks with and without a shared prompt ("Worked Example 2", answer A5);
* per-token KV bytes 2 * L * H * d_k * sizeof(dtype) and the utilisation bound
  eta_paged >= 1 - (B - 1) / L ("Paged Attention and vLLM", "KV Cache
  Fundamentals" and "Memory Efficiency: Fragmentation Analysis").
"""
from __future__ import annotations

from fractions import Fraction


def blocks_for(tokens: int, block_size: int) -> int:
    """Number of B-token blocks that hold `tokens` tokens (ceiling division)."""
    if tokens < 0 or block_size <= 0:
        raise ValueError("tokens >= 0 and block_size > 0 required")
    return (tokens + block_size - 1) // block_size


def fragmentation(lengths, block_size: int, max_len: int) -> dict:
    """Paged (block-rounded) versus contiguous max_len reservation for a batch."""
    blocks = [blocks_for(n, block_size) for n in lengths]
    tokens = sum(lengths)
    paged = sum(blocks) * block_size
    naive = max_len * len(lengths)
    return {
        "blocks": blocks,
        "total_blocks": sum(blocks),
        "tokens": tokens,
        "paged_slots": paged,
        "naive_slots": naive,
        "paged_waste": paged - tokens,
        "naive_waste": naive - tokens,
        "paged_frag": Fraction(paged - tokens, paged),
        "naive_frag": Fraction(naive - tokens, naive),
        "reduction": Fraction(naive, paged),
    }


def shared_prompt_blocks(prompt: int, suffix: int, block_size: int, requests: int,
                         share_partial: bool) -> dict:
    """Blocks for `requests` requests of prompt+suffix tokens, unshared versus shared.

    Without sharing each request stores its prompt and its suffix in separate
    block runs.  With sharing the prompt's blocks are stored once; when
    ``share_partial`` is false only the prompt's *full* blocks are shared and
    the straddling block is stored per request.
    """
    per_req_unshared = blocks_for(prompt, block_size) + blocks_for(suffix, block_size)
    without = per_req_unshared * requests
    if share_partial:
        shared = blocks_for(prompt, block_size)
        private = blocks_for(suffix, block_size)
    else:
        shared = prompt // block_size
        private = blocks_for(prompt - shared * block_size + suffix, block_size)
    with_sharing = shared + private * requests
    return {"per_request_unshared": per_req_unshared, "without": without,
            "shared_blocks": shared, "private_per_request": private,
            "with": with_sharing, "reduction": Fraction(without, with_sharing)}


def full_shareable_blocks(prompt: int, block_size: int) -> int:
    """Blocks lying entirely inside the prompt (only these can be shared as-is)."""
    return prompt // block_size


def kv_bytes_per_token(layers: int, heads: int, head_dim: int, dtype_bytes: int) -> int:
    """M_token = 2 (K and V) * L * H * d_k * sizeof(dtype)."""
    return 2 * layers * heads * head_dim * dtype_bytes


def eta_paged(lengths, block_size: int) -> Fraction:
    """Fraction of reserved paged slots that hold tokens."""
    tokens = sum(lengths)
    slots = sum(blocks_for(n, block_size) for n in lengths) * block_size
    return Fraction(tokens, slots) if slots else Fraction(1)


def eta_paged_lower_bound(mean_len, block_size: int) -> Fraction:
    """1 - (B - 1) / L, the page's lower bound on a sequence's utilisation."""
    return 1 - Fraction(block_size - 1) / Fraction(mean_len)
