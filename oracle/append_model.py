"""Plain-Python model of the K/V append step (test oracle).

"feat: add paged-attention monolithic decode-only AR foundation" (lucebox
pull 555), Summary: the paging metadata (block table and sequence lengths)
stays resident on the device next to the K/V pool, and a decode step uploads
only the 4-byte id of each fresh 16-token block instead of the whole table.
Validation exercises "prefill -> many block boundaries".  This model restates
one append step on host arrays, one sequence at a time:

- the new token of sequence s goes to position L = lens[s]: table entry
  j = L // B, slot L % B;
- when the slot is 0 the token starts a block: table[s][j] = fresh[s] (the
  caller allocated that block and uploaded its id); otherwise the block is
  the one already in table[s][j];
- every K/V head's new row is quantised (oracle.quantize_row) into that slot
  of that block, and lens[s] becomes L + 1;
- a table with no entry j left, or a block id outside [0, n_pool_blocks),
  leaves the sequence untouched and sets a status bit (the library's values,
  restated: 1 = block id outside the pool, 8 = table full).

TEST INFRASTRUCTURE ONLY: the product path never imports this."""
import numpy as np

from . import quantize_row

STATUS_CORRUPT_TABLE = 1
STATUS_APPEND_RANGE = 8


def append(pool_k: np.ndarray, pool_v: np.ndarray, table: np.ndarray, lens: np.ndarray,
           k_new: np.ndarray, v_new: np.ndarray, fresh: np.ndarray, *, block_size: int,
           k_type: int, v_type: int) -> int:
    """pool_k / pool_v: uint8 [n_blocks, B, hkv, row]; table: int32 [S, stride];
    lens: int32 [S]; k_new / v_new: float32 [S, hkv, d]; fresh: int32 [S].
    Updates the arrays in place and returns the status bits."""
    n_blocks, _, hkv, _ = pool_k.shape
    S, stride = table.shape
    status = 0
    for s in range(S):
        L = int(lens[s])
        if L < 0:
            status |= STATUS_APPEND_RANGE
            continue
        j, slot = divmod(L, block_size)
        if j >= stride:
            status |= STATUS_APPEND_RANGE
            continue
        blk = int(fresh[s]) if slot == 0 else int(table[s, j])
        if not 0 <= blk < n_blocks:
            status |= STATUS_CORRUPT_TABLE
            continue
        if slot == 0:
            table[s, j] = blk
        for g in range(hkv):
            pool_k[blk, slot, g] = quantize_row(k_type, k_new[s, g])
            pool_v[blk, slot, g] = quantize_row(v_type, v_new[s, g])
        lens[s] = L + 1
    return status
