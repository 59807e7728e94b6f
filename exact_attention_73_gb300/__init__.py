"""libattn for GB300: exact fused attention behind a C ABI.

``binding`` holds the Python names of the C entry points; ``build`` compiles
the CUDA library in-tree; ``inputs`` holds the seeded synthetic inputs.
"""
