"""Float64 CPU oracle for two-copy block-diffusion attention.

Test infrastructure only: the product library never imports this package.
"""
