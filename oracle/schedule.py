"""Tile-grid, mask and program-order arithmetic -- TEST INFRASTRUCTURE ONLY.

Plain Python restatements of the integer arithmetic the pages print, used to
check the GPU library's scheduler and edge handling.  Nothing here imports the
product package.
"""
from __future__ import annotations


def cdiv(a: int, b: int) -> int:
    """Ceiling division, the grid size rule of "I Wrote a GPU Matmul Kernel From
    Scratch in Triton", Step 3 (1023 rows with BLOCK_SIZE 64 give 16 blocks)."""
    return -(-a // b)


def grid_2d(M: int, N: int, block_m: int, block_n: int) -> tuple[int, int]:
    """Programs along rows and columns of C: one per output tile ("Writing GPU
    kernels in Triton", section 3.2: C of 96x80 with 32x32 tiles gives (3, 3))."""
    return cdiv(M, block_m), cdiv(N, block_n)


def k_rounds(K: int, block_k: int) -> int:
    """K-loop trip count of one program (section 3.3/3.4 of the same page)."""
    return cdiv(K, block_k)


def row_major_tile(pid: int, num_blocks_n: int) -> tuple[int, int]:
    """1-D program id -> (tile row, tile column) in row-major order, as in the
    teaching kernel of "Triton 04: Matmul, Autotune and PyTorch integration"."""
    return pid // num_blocks_n, pid % num_blocks_n


def group_major_tile(pid: int, num_blocks_m: int, num_blocks_n: int, group: int) -> tuple[int, int]:
    """1-D program id -> (tile row, tile column) in group-major order.

    Step 4 of "I Wrote a GPU Matmul Kernel From Scratch in Triton": programs
    are taken in strips of ``group`` tile rows; inside a strip consecutive ids
    walk down a column first and then move one column right.  The last strip
    is only as tall as the tile rows that remain (the min() of that step).
    """
    per_group = group * num_blocks_n
    group_id = pid // per_group
    first_row = group_id * group
    height = min(num_blocks_m - first_row, group)
    local = pid % per_group
    return first_row + local % height, local // height


def order_layout(num_blocks_m: int, num_blocks_n: int, group: int | None) -> list[list[int]]:
    """layout[row][col] = the program id that computes tile (row, col).

    ``group=None`` gives the row-major order, otherwise the group-major order.
    """
    layout = [[-1] * num_blocks_n for _ in range(num_blocks_m)]
    for pid in range(num_blocks_m * num_blocks_n):
        if group is None:
            r, c = row_major_tile(pid, num_blocks_n)
        else:
            r, c = group_major_tile(pid, num_blocks_m, num_blocks_n, group)
        layout[r][c] = pid
    return layout


def out_of_range(extent: int, block: int) -> int:
    """Masked positions in the last block along one dimension (section 4.6 of
    "Writing GPU kernels in Triton": 70 rows in 32-row tiles leave 26 masked)."""
    return cdiv(extent, block) * block - extent
